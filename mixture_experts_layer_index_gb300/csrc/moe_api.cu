// C ABI (include/moe.h): argument validation, workspace planning, path choice
// and the ordered, sync-free launch sequence of each entry point.  It plays the
// role of the entry layer described in the Code changes of "perf: add
// small-batch route MMA for MoE": choosing the small-batch path, picking the
// K split, laying out one workspace, checking every argument, and writing into
// an output the caller allocated.
#include <cstddef>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "common.cuh"
#include "internal.h"

namespace moe {

// ------------------------------------------------------------------ device queries
EncodeTiledFn get_encode_tiled() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

int num_sms() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cache[dev] == 0) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cache[dev] = v;
  }
  return cache[dev];
}

// ------------------------------------------------------------------ stage timing
namespace {
struct StageRecord {
  int stage;
  cudaEvent_t begin, end;
};
struct Profiler {
  std::mutex mu;
  bool on = false;
  std::string only;  // time only this stage ("" = every stage)
  std::vector<std::string> names;
  std::vector<StageRecord> records;
  std::vector<cudaEvent_t> pool;
  int open = -1;  // index of the record whose end is pending
  cudaEvent_t take() {
    if (!pool.empty()) {
      cudaEvent_t e = pool.back();
      pool.pop_back();
      return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
  }
  void recycle() {
    for (auto& r : records) {
      if (r.begin) pool.push_back(r.begin);
      if (r.end) pool.push_back(r.end);
    }
    records.clear();
    names.clear();
    open = -1;
  }
};
Profiler& prof() {
  static Profiler p;
  return p;
}
bool capturing(cudaStream_t s) {
  cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &st) != cudaSuccess) return true;
  return st != cudaStreamCaptureStatusNone;
}
}  // namespace

void stage_begin(const char* name, cudaStream_t s) {
  Profiler& P = prof();
  std::lock_guard<std::mutex> lk(P.mu);
  if (!P.on || capturing(s)) return;
  if (!P.only.empty() && P.only != name) return;
  int idx = -1;
  for (size_t i = 0; i < P.names.size(); ++i)
    if (P.names[i] == name) idx = static_cast<int>(i);
  if (idx < 0) {
    P.names.emplace_back(name);
    idx = static_cast<int>(P.names.size()) - 1;
  }
  StageRecord r{idx, P.take(), P.take()};
  if (!r.begin || !r.end || cudaEventRecord(r.begin, s) != cudaSuccess) {
    if (r.begin) P.pool.push_back(r.begin);
    if (r.end) P.pool.push_back(r.end);
    return;
  }
  P.records.push_back(r);
  P.open = static_cast<int>(P.records.size()) - 1;
}

void stage_end(cudaStream_t s) {
  Profiler& P = prof();
  std::lock_guard<std::mutex> lk(P.mu);
  if (!P.on || P.open < 0) return;
  if (cudaEventRecord(P.records[P.open].end, s) != cudaSuccess) {
    P.records[P.open].stage = -1;
  }
  P.open = -1;
}

// ------------------------------------------------------------------ planning
static bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

ShuffleLayout plan_shuffle(int T, int E, int k, size_t base) {
  ShuffleLayout L;
  const size_t R = static_cast<size_t>(T) * k;
  const int TB = route_tokens_per_block(k);
  L.nblk = T > 0 ? (T + TB - 1) / TB : 0;
  size_t off = base;
  L.lrank = off;
  off = align_up(off + R * 4, 256);
  L.blockcounts = off;
  off = align_up(off + static_cast<size_t>(L.nblk) * E * 4, 256);
  L.tile_scratch = off;
  off = align_up(off + static_cast<size_t>(E + 1) * 4, 256);
  L.total = off;
  return L;
}

// Largest T for which AUTO takes the route-direct path (beyond it, the grouped
// path), per FP8 mode.  Measured on GB300 with both paths captured in CUDA
// graphs, L2 flushed between calls, k = 8: per-tensor (E=192, H=4096, I=192)
// route-direct is faster through T=96 (156.8 vs 166.7 us), even at T=112 and
// slower at T=128; blockwise (E=128, H=2048, I=768 / H=4096, I=512)
// route-direct is faster through T=64 (140.4 vs 144.5 / 183.4 vs 189.6 us) and
// even or slower at T=96.
constexpr int kAutoRouteDirectMaxTokensPerTensor = 96;
constexpr int kAutoRouteDirectMaxTokensBlockwise = 64;

// S shared experts run on the grouped path only (their rows join the expert-sorted
// intermediate tensors and the tile map).
static moe_path resolve_path(const moe_problem& p, int S = 0) {
  if (p.path != MOE_PATH_AUTO) return p.path;
  if (p.quant == MOE_BF16 || p.quant == MOE_MXFP8 || S > 0) return MOE_PATH_GROUPED;
  const int limit = p.quant == MOE_FP8_BLOCK128 ? kAutoRouteDirectMaxTokensBlockwise
                                                : kAutoRouteDirectMaxTokensPerTensor;
  if (p.T > limit || static_cast<long long>(p.T) * p.k > kRouteDirectMaxRoutes) return MOE_PATH_GROUPED;
  return MOE_PATH_ROUTE_DIRECT;
}

// Number of K splits of the route-direct Gate/Up: the K slice of one work item
// (H / splits bytes, a multiple of 128) at most 1024 bytes, so that two CTAs'
// weight stages and 8-token x slices fit in one SM's shared memory, then
// doubled while the items (distinct experts x 64-row blocks x splits, at most)
// number fewer than three per SM of a 152-SM part and the slice stays at least
// 512 bytes long.  Depends only on the shape, so the workspace size is a pure
// function of the problem.
static int route_direct_splits(const moe_problem& p) {
  const int R = p.T * p.k;
  const int maxU = R < p.E ? R : p.E;
  const long long items = static_cast<long long>(maxU) * (2 * p.I / 64);
  int s = 1;
  while (p.H / s > 1024 && (p.H / (2 * s)) % 128 == 0) s *= 2;
  while (items * s < 3 * 152 && (p.H / (2 * s)) % 128 == 0 && p.H / (2 * s) >= 512) s *= 2;
  return s;
}

static moe_status validate_shape(const moe_problem& p, int S = 0) {
  if (p.T < 0 || p.E < 1 || p.k < 1 || p.H < 1 || p.I < 1) return MOE_ERR_INVALID_ARG;
  if (p.k > p.E) return MOE_ERR_INVALID_ARG;
  if (p.quant != MOE_BF16 && p.quant != MOE_FP8_PER_TENSOR && p.quant != MOE_FP8_BLOCK128 && p.quant != MOE_MXFP8)
    return MOE_ERR_INVALID_ARG;
  if (p.path != MOE_PATH_AUTO && p.path != MOE_PATH_GROUPED && p.path != MOE_PATH_ROUTE_DIRECT)
    return MOE_ERR_INVALID_ARG;
  if (p.E > kMaxE || p.k > kMaxK) return MOE_ERR_UNSUPPORTED;
  if (static_cast<long long>(p.T) * p.k >= (1ll << 31)) return MOE_ERR_UNSUPPORTED;
  if (static_cast<long long>(p.E) * 2 * p.I >= (1ll << 31) || static_cast<long long>(p.E) * p.H >= (1ll << 31))
    return MOE_ERR_UNSUPPORTED;
  if (p.quant == MOE_BF16) {
    if (p.H % 64 || p.I % 64) return MOE_ERR_UNSUPPORTED;
  } else if (p.quant == MOE_FP8_PER_TENSOR) {
    if (p.H % 64 || p.I % 64) return MOE_ERR_UNSUPPORTED;
  } else {  // blockwise FP8 (x scales per 128 columns of H) and MXFP8
    if (p.H % 128 || p.I % 64) return MOE_ERR_UNSUPPORTED;
  }
  if (S < 0) return MOE_ERR_INVALID_ARG;
  if (S > kMaxShared) return MOE_ERR_UNSUPPORTED;
  if (static_cast<long long>(p.T) * (p.k + S) >= (1ll << 31)) return MOE_ERR_UNSUPPORTED;
  const moe_path path = resolve_path(p, S);
  if (path == MOE_PATH_ROUTE_DIRECT) {
    if (p.quant == MOE_BF16 || p.quant == MOE_MXFP8 || S > 0) return MOE_ERR_UNSUPPORTED;

    if (static_cast<long long>(p.T) * p.k > kRouteDirectMaxRoutes) return MOE_ERR_UNSUPPORTED;
    // shared-memory staging of one work item's operand rows
    if (p.I > 4096 || p.H / route_direct_splits(p) > 4096) return MOE_ERR_UNSUPPORTED;
  }
  return MOE_OK;
}

bool plan_forward(const moe_problem& p, ForwardLayout* out, int S) {
  if (validate_shape(p, S) != MOE_OK) return false;
  ForwardLayout L;
  L.path = resolve_path(p, S);
  const size_t T = p.T, E = p.E, k = p.k, H = p.H, I = p.I, R = T * k;
  // rows of the intermediate tensors: the routes, then T rows per shared expert
  const size_t RS = R + static_cast<size_t>(S) * T;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes, 256);
    return at;
  };
  L.header = take(sizeof(DeviceHeader));
  L.ids = take(R * 4);
  L.w = take(R * 4);
  if (L.path == MOE_PATH_GROUPED) {
    L.shuf = plan_shuffle(p.T, p.E, p.k, off);
    off = L.shuf.total;
    L.counts = take(E * 4);
    L.offsets = take((E + 1) * 4);
    L.perm = take(R * 4);
    L.inv = take(R * 4);
    L.max_tiles = static_cast<int>(R / kGemmBM + E + static_cast<size_t>(S) * ((T + kGemmBM - 1) / kGemmBM));
    L.tiles = take(static_cast<size_t>(L.max_tiles) * 16);
    L.num_tiles = take(16);
    const size_t eb = p.quant == MOE_BF16 ? 2 : 1;  // bytes per element of the GEMM inputs
    L.xs = take(RS * H * eb);
    if (p.quant == MOE_FP8_BLOCK128) L.xs_scale = take(RS * (H / 128) * 4);
    if (p.quant == MOE_FP8_PER_TENSOR) L.abf = take(RS * I * 2);
    L.h = take(RS * I * eb);
    if (p.quant == MOE_FP8_BLOCK128) L.sh = take(RS * ((I + 127) / 128) * 4);
    if (p.quant == MOE_MXFP8) {
      const int Hc = p.H / 32, Ic = p.I / 32;
      L.xs_sc = take(RS * Hc);
      L.xs_sf = take(mx_blocked_bytes(L.max_tiles, Hc));
      L.h_sf = take(mx_blocked_bytes(L.max_tiles, Ic));
      L.padbase = take((E + S) * 4);
      L.w1_sf = take(mx_blocked_bytes(E * ((I + 95) / 96) * 2, Hc));  // two blocks per Gate/Up unit
      L.w2_sf = take(mx_blocked_bytes(E * ((H + 191) / 192) * 2, Ic));  // two blocks per Down unit
      if (S > 0) {
        L.w1s_sf = take(mx_blocked_bytes(static_cast<size_t>(S) * ((I + 95) / 96) * 2, Hc));
        L.w2s_sf = take(mx_blocked_bytes(static_cast<size_t>(S) * ((H + 191) / 192) * 2, Ic));
      }
    }
    L.o = take(RS * H * 2);
  } else {
    L.splits = route_direct_splits(p);
    L.xq = take(T * H);
    L.sx = take(p.quant == MOE_FP8_BLOCK128 ? T * (H / 128) * 4 : 16);
    L.uniq = take(route_direct_uniq_bytes(p.T, p.E, p.k));
    L.part = take(static_cast<size_t>(L.splits) * R * 2 * I * 4);
    L.act = take(R * I * 4);
    L.sh = take(p.quant == MOE_FP8_BLOCK128 ? R * ((I + 127) / 128) * 4 : 16);
    L.o = take(R * H * 4);
  }
  L.total = off;
  *out = L;
  return true;
}

template <typename Ptr>
static Ptr at(void* ws, size_t off) {
  return reinterpret_cast<Ptr>(static_cast<uint8_t*>(ws) + off);
}

static moe_status from_cuda(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// How the Gate/Up GEMM obtains its expert-sorted activation rows.  Default: the
// scatter kernel copies every route's x row to its sorted position and the GEMM
// loads contiguous TMA tiles.  MOE_GATEUP_A=gather4 (environment, read once)
// selects the fully fused variant that gathers x rows inside the GEMM with TMA
// tile::gather4 instead; it is kept for comparison (it measured 3.2x slower per
// K stage on GB300).
static bool gateup_gather4() {
  static const bool v = [] {
    const char* e = std::getenv("MOE_GATEUP_A");
    return e && std::strcmp(e, "gather4") == 0;
  }();
  return v;
}

}  // namespace moe

using namespace moe;

extern "C" {

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported problem (outside this library's limits)";
    case MOE_ERR_WORKSPACE: return "workspace missing or too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_DEVICE_TIMEOUT: return "device-side bounded wait timed out";
    case MOE_ERR_DEVICE_BOUNDS: return "device-side index out of range";
  }
  return "unknown status";
}

moe_status moe_route(const float* scores, int T, int E, int k, int32_t* ids, float* w, moe_stream_t stream) {
  if (T < 0 || E < 1 || k < 1 || k > E) return MOE_ERR_INVALID_ARG;
  if (E > kMaxE || k > kMaxK || static_cast<long long>(T) * k >= (1ll << 31)) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!scores || !ids || !w || !aligned(scores, 4) || !aligned(ids, 4) || !aligned(w, 4)) return MOE_ERR_INVALID_ARG;
  return from_cuda(launch_route_rank(scores, nullptr, T, E, k, ids, w, nullptr, nullptr, nullptr, true, false,
                                     reinterpret_cast<cudaStream_t>(stream)));
}

size_t moe_shuffle_workspace_size(int T, int E, int k) {
  if (T < 0 || E < 1 || k < 1 || E > kMaxE || k > kMaxK) return 0;
  return plan_shuffle(T, E, k, align_up(sizeof(DeviceHeader), 256)).total;
}

moe_status moe_shuffle(const int32_t* ids, int T, int E, int k, int32_t* counts, int32_t* offsets, int32_t* perm,
                       int32_t* inv, void* ws, size_t ws_bytes, moe_stream_t stream) {
  if (T < 0 || E < 1 || k < 1 || k > E) return MOE_ERR_INVALID_ARG;
  if (E > kMaxE || k > kMaxK || static_cast<long long>(T) * k >= (1ll << 31)) return MOE_ERR_UNSUPPORTED;
  if (!counts || !offsets || !aligned(counts, 4) || !aligned(offsets, 4)) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!ids || !perm || !inv || !aligned(ids, 4) || !aligned(perm, 4) || !aligned(inv, 4)))
    return MOE_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, 16)) return MOE_ERR_WORKSPACE;
  const ShuffleLayout L = plan_shuffle(T, E, k, align_up(sizeof(DeviceHeader), 256));
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  DeviceHeader* hdr = at<DeviceHeader*>(ws, 0);
  cudaError_t e = launch_reset_header(hdr, s);
  if (e == cudaSuccess && T == 0) {
    e = cudaMemsetAsync(counts, 0, static_cast<size_t>(E) * 4, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(offsets, 0, static_cast<size_t>(E + 1) * 4, s);
    return from_cuda(e);
  }
  int32_t* lrank = at<int32_t*>(ws, L.lrank);
  int32_t* bc = at<int32_t*>(ws, L.blockcounts);
  if (e == cudaSuccess)
    e = launch_route_rank(nullptr, ids, T, E, k, nullptr, nullptr, lrank, bc, hdr, false, true, s);
  if (e == cudaSuccess)
    e = launch_scan_tiles(bc, L.nblk, E, counts, offsets, nullptr, nullptr, 0, kGemmBM, nullptr, hdr, s);
  if (e == cudaSuccess) e = launch_scatter(ids, lrank, bc, T, E, k, perm, inv, s);
  return from_cuda(e);
}

moe_status moe_tile_map(const int32_t* counts, int E, int BM, int32_t* tiles, int32_t* num_tiles, int max_tiles,
                        void* ws, size_t ws_bytes, moe_stream_t stream) {
  if (E < 1 || BM < 1 || BM > 1024 || max_tiles < 0) return MOE_ERR_INVALID_ARG;
  if (E > kMaxE) return MOE_ERR_UNSUPPORTED;
  if (!counts || !num_tiles || (max_tiles > 0 && !tiles) || !aligned(counts, 4) || !aligned(num_tiles, 4) ||
      !aligned(tiles, 16))
    return MOE_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, 16)) return MOE_ERR_WORKSPACE;
  if (ws_bytes < moe_shuffle_workspace_size(0, E, 1)) return MOE_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  DeviceHeader* hdr = at<DeviceHeader*>(ws, 0);
  cudaError_t e = launch_reset_header(hdr, s);
  if (e == cudaSuccess) e = launch_tile_map(counts, E, BM, tiles, num_tiles, max_tiles, nullptr, hdr, s);
  return from_cuda(e);
}

moe_path moe_select_path(const moe_problem* p) {
  if (!p) return MOE_PATH_AUTO;
  return resolve_path(*p);
}

size_t moe_workspace_size(const moe_problem* p) {
  if (!p) return 0;
  ForwardLayout L;
  if (!plan_forward(*p, &L)) return 0;
  return L.total;
}

moe_status moe_forward(const moe_problem* pp, const void* x, const float* scores, const void* w1, const void* w2,
                       const float* w1_scale, const float* w2_scale, void* y, void* ws, size_t ws_bytes,
                       moe_stream_t stream) {
  return moe_forward_ex(pp, nullptr, x, scores, w1, w2, w1_scale, w2_scale, y, ws, ws_bytes, stream);
}

size_t moe_workspace_size_ex(const moe_problem* p, const moe_forward_options* opt) {
  if (!p) return 0;
  ForwardLayout L;
  if (!plan_forward(*p, &L, opt ? opt->n_shared : 0)) return 0;
  return L.total;
}

moe_status moe_forward_ex(const moe_problem* pp, const moe_forward_options* opt, const void* x, const float* scores,
                          const void* w1, const void* w2, const float* w1_scale, const float* w2_scale, void* y,
                          void* ws, size_t ws_bytes, moe_stream_t stream) {
  if (!pp) return MOE_ERR_INVALID_ARG;
  const moe_problem p = *pp;
  const moe_forward_options o = opt ? *opt : moe_forward_options{};
  const int S = o.n_shared;
  if (o.y_fp32 != 0 && o.y_fp32 != 1) return MOE_ERR_INVALID_ARG;
  if (o.mx_weight_scales_blocked != 0 && (o.mx_weight_scales_blocked != 1 || p.quant != MOE_MXFP8))
    return MOE_ERR_INVALID_ARG;
  if (o.mx_weight_scales_blocked && (!aligned(w1_scale, 16) || !aligned(w2_scale, 16))) return MOE_ERR_INVALID_ARG;
  const moe_status vs = validate_shape(p, S);
  if (vs != MOE_OK) return vs;
  if (p.T == 0) return MOE_OK;
  if (!x || !scores || !w1 || !w2 || !y) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(w1, 16) || !aligned(w2, 16) || !aligned(y, 16) || !aligned(scores, 4))
    return MOE_ERR_INVALID_ARG;
  if (p.quant == MOE_BF16) {
    if (w1_scale || w2_scale) return MOE_ERR_INVALID_ARG;
  } else {
    if (!w1_scale || !w2_scale || !aligned(w1_scale, 4) || !aligned(w2_scale, 4)) return MOE_ERR_INVALID_ARG;
  }
  if (S > 0) {
    if (!o.w1_shared || !o.w2_shared || !aligned(o.w1_shared, 16) || !aligned(o.w2_shared, 16))
      return MOE_ERR_INVALID_ARG;
    if (p.quant == MOE_BF16) {
      if (o.w1_shared_scale || o.w2_shared_scale) return MOE_ERR_INVALID_ARG;
    } else if (!o.w1_shared_scale || !o.w2_shared_scale || !aligned(o.w1_shared_scale, 4) ||
               !aligned(o.w2_shared_scale, 4)) {
      return MOE_ERR_INVALID_ARG;
    }
  }
  ForwardLayout L;
  if (!plan_forward(p, &L, S)) return MOE_ERR_UNSUPPORTED;
  if (!ws || !aligned(ws, 256)) return MOE_ERR_WORKSPACE;
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  DeviceHeader* hdr = at<DeviceHeader*>(ws, L.header);
  int32_t* ids = at<int32_t*>(ws, L.ids);
  float* w = at<float*>(ws, L.w);
  cudaError_t e = cudaSuccess;
  if (L.path == MOE_PATH_GROUPED) {
    int32_t* lrank = at<int32_t*>(ws, L.shuf.lrank);
    int32_t* bc = at<int32_t*>(ws, L.shuf.blockcounts);
    int32_t* counts = at<int32_t*>(ws, L.counts);
    int32_t* offsets = at<int32_t*>(ws, L.offsets);
    int32_t* perm = at<int32_t*>(ws, L.perm);
    int32_t* inv = at<int32_t*>(ws, L.inv);
    int32_t* tiles = at<int32_t*>(ws, L.tiles);
    int32_t* num_tiles = at<int32_t*>(ws, L.num_tiles);
    e = launch_reset_header(hdr, s);
    if (e == cudaSuccess)
      e = launch_route_rank(scores, nullptr, p.T, p.E, p.k, ids, w, lrank, bc, hdr, true, true, s,
                            p.quant == MOE_FP8_PER_TENSOR ? x : nullptr, static_cast<size_t>(p.T) * p.H);
    if (e == cudaSuccess)
      e = launch_scan_tiles(bc, L.shuf.nblk, p.E, counts, offsets, tiles, num_tiles, L.max_tiles, kGemmBM, nullptr,
                            hdr, s, p.T, S, p.T * p.k, p.quant == MOE_MXFP8 ? at<int32_t*>(ws, L.padbase) : nullptr);
    const bool f8 = p.quant == MOE_FP8_PER_TENSOR;
    const bool blockwise = p.quant == MOE_FP8_BLOCK128;
    const bool mxfp8 = p.quant == MOE_MXFP8;
    // the variant that gathers x inside the GEMM reads routed rows only
    const bool gather4 = p.quant == MOE_BF16 && S == 0 && gateup_gather4();
    void* xs = at<void*>(ws, L.xs);
    float* xs_scale = blockwise ? at<float*>(ws, L.xs_scale) : nullptr;
    float* sh = blockwise ? at<float*>(ws, L.sh) : nullptr;
    if (e == cudaSuccess) {
      if (mxfp8)
        e = launch_scatter_gather_mx(ids, lrank, bc, p.T, p.E, p.k, p.H, x, xs, at<uint8_t*>(ws, L.xs_sc),
                                     at<uint8_t*>(ws, L.xs_sf), at<int32_t*>(ws, L.padbase), perm, inv, s, S);
      else if (f8)
        e = launch_scatter_gather_q(ids, lrank, bc, p.T, p.E, p.k, p.H, x, xs, perm, inv, hdr, s, S);
      else if (blockwise)
        e = launch_scatter_gather_qb(ids, lrank, bc, p.T, p.E, p.k, p.H, x, xs, xs_scale, perm, inv, s, S);
      else if (gather4)
        e = launch_scatter(ids, lrank, bc, p.T, p.E, p.k, perm, inv, s);
      else
        e = launch_scatter_gather(ids, lrank, bc, p.T, p.E, p.k, p.H, x, xs, perm, inv, s, S);
    }
    if (e == cudaSuccess) {
      GroupedArgs g{};
      g.T = p.T; g.E = p.E; g.k = p.k; g.H = p.H; g.I = p.I;
      g.R = p.T * p.k + S * p.T;
      g.x = x; g.w1 = w1; g.w2 = w2;
      g.S = S;
      g.w1s = o.w1_shared; g.w2s = o.w2_shared;
      g.w1s_scale = o.w1_shared_scale; g.w2s_scale = o.w2_shared_scale;
      g.f8 = f8 || blockwise;
      g.w1_scale = w1_scale;
      g.w2_scale = w2_scale;
      g.a_bf16 = f8 ? at<void*>(ws, L.abf) : nullptr;
      if (mxfp8) g.f8 = true;
      g.xs = gather4 ? nullptr : xs;
      g.perm = perm; g.tiles = tiles; g.num_tiles = num_tiles; g.max_tiles = L.max_tiles;
      g.h = at<void*>(ws, L.h);
      g.o = at<void*>(ws, L.o);
      g.hdr = hdr;
      if (mxfp8) {
        uint8_t* xs_sf = at<uint8_t*>(ws, L.xs_sf);
        uint8_t* h_sf = at<uint8_t*>(ws, L.h_sf);
        uint8_t* w1_sf = at<uint8_t*>(ws, L.w1_sf);
        uint8_t* w2_sf = at<uint8_t*>(ws, L.w2_sf);
        uint8_t* w1s_sf = S > 0 ? at<uint8_t*>(ws, L.w1s_sf) : nullptr;
        uint8_t* w2s_sf = S > 0 ? at<uint8_t*>(ws, L.w2s_sf) : nullptr;
        if (o.mx_weight_scales_blocked) {  // converted once by the caller
          w1_sf = const_cast<uint8_t*>(reinterpret_cast<const uint8_t*>(w1_scale));
          w2_sf = const_cast<uint8_t*>(reinterpret_cast<const uint8_t*>(w2_scale));
          if (S > 0) {
            w1s_sf = const_cast<uint8_t*>(reinterpret_cast<const uint8_t*>(o.w1_shared_scale));
            w2s_sf = const_cast<uint8_t*>(reinterpret_cast<const uint8_t*>(o.w2_shared_scale));
          }
        } else {
          e = launch_mx_blocked_weights(reinterpret_cast<const uint8_t*>(w1_scale),
                                        reinterpret_cast<const uint8_t*>(w2_scale), p.E, p.H, p.I, w1_sf, w2_sf, s);
          if (e == cudaSuccess && S > 0)
            e = launch_mx_blocked_weights(reinterpret_cast<const uint8_t*>(o.w1_shared_scale),
                                          reinterpret_cast<const uint8_t*>(o.w2_shared_scale), S, p.H, p.I, w1s_sf,
                                          w2s_sf, s);
        }
        if (e == cudaSuccess) e = launch_gateup_mx(g, xs_sf, w1_sf, w1s_sf, h_sf, s);
        if (e == cudaSuccess) e = launch_down_mx(g, h_sf, w2_sf, w2s_sf, s);
      } else if (blockwise) {
        e = launch_gateup_blockwise(g, xs_scale, sh, s);
        if (e == cudaSuccess) e = launch_down_blockwise(g, sh, s);
      } else {
        e = launch_gateup_bf16(g, s);
        if (e == cudaSuccess && f8)
          e = launch_quant_rows(g.a_bf16, g.h, static_cast<size_t>(g.R) * p.I, hdr, s);
        if (e == cudaSuccess) e = launch_down_bf16(g, s);
      }
    }
    if (e == cudaSuccess) {
      CombineArgs c{p.T, p.k, p.H, at<void*>(ws, L.o), false, w, y, inv};
      c.S = S;
      c.y_f32 = o.y_fp32 != 0;
      e = launch_combine(c, s);
    }
  } else {
    DecodeArgs d{};
    d.T = p.T; d.E = p.E; d.k = p.k; d.H = p.H; d.I = p.I; d.R = p.T * p.k;
    d.quant = p.quant;
    d.x = x; d.scores = scores;
    d.w1 = static_cast<const uint8_t*>(w1);
    d.w2 = static_cast<const uint8_t*>(w2);
    d.w1_scale = w1_scale; d.w2_scale = w2_scale;
    d.ids = ids; d.w = w;
    d.xq = at<uint8_t*>(ws, L.xq);
    d.sx = at<float*>(ws, L.sx);
    d.uniq = at<int32_t*>(ws, L.uniq);
    d.part = at<float*>(ws, L.part);
    d.act = at<void*>(ws, L.act);
    d.sh = at<float*>(ws, L.sh);
    d.o = at<float*>(ws, L.o);
    d.splits = L.splits;
    d.hdr = hdr;
    e = launch_route_direct(d, s);
    if (e == cudaSuccess) {
      CombineArgs c{p.T, p.k, p.H, d.o, true, w, y, nullptr};
      c.y_f32 = o.y_fp32 != 0;
      e = launch_combine_pdl(c, s);
    }
  }
  return from_cuda(e);
}

size_t moe_mx_weight_scales_bytes(int E, int H, int I, int which) {
  if (E < 1 || H < 1 || I < 1 || H % 128 || I % 64 || (which != 1 && which != 2)) return 0;
  return which == 1 ? mx_blocked_bytes(static_cast<size_t>(E) * ((I + 95) / 96) * 2, H / 32)
                    : mx_blocked_bytes(static_cast<size_t>(E) * ((H + 191) / 192) * 2, I / 32);
}

moe_status moe_mx_weight_scales(const uint8_t* w1_scale, const uint8_t* w2_scale, int E, int H, int I,
                                uint8_t* w1_blocked, uint8_t* w2_blocked, moe_stream_t stream) {
  if (E < 1 || H < 1 || I < 1) return MOE_ERR_INVALID_ARG;
  if (E > kMaxE || H % 128 || I % 64 || static_cast<long long>(E) * 2 * I * H >= (1ll << 40)) return MOE_ERR_UNSUPPORTED;
  if (!w1_scale || !w2_scale || !w1_blocked || !w2_blocked || !aligned(w1_scale, 4) || !aligned(w2_scale, 4) ||
      !aligned(w1_blocked, 16) || !aligned(w2_blocked, 16))
    return MOE_ERR_INVALID_ARG;
  return from_cuda(launch_mx_blocked_weights(w1_scale, w2_scale, E, H, I, w1_blocked, w2_blocked,
                                             reinterpret_cast<cudaStream_t>(stream)));
}

size_t moe_mx_blocked_bytes(int rows, int cols, int groups) {
  if (rows < 0 || cols < 1 || groups < 1) return 0;
  return mx_blocked_bytes(static_cast<size_t>(rows) / kGemmBM + groups, cols);
}

static constexpr int kMxMaxGroups = 4096;

size_t moe_mx_blocked_workspace_size(int rows, int groups) {
  if (rows < 0 || groups < 1 || groups > kMxMaxGroups) return 0;
  const size_t max_tiles = static_cast<size_t>(rows) / kGemmBM + groups;
  return align_up(sizeof(DeviceHeader), 256) + align_up(max_tiles * 16, 256) + 256;
}

moe_status moe_mx_blocked_scales(const uint8_t* scales, int rows, int cols, const int32_t* group_offsets, int groups,
                                 uint8_t* out, size_t out_bytes, int32_t* group_starts, void* ws, size_t ws_bytes,
                                 moe_stream_t stream) {
  if (rows < 0 || cols < 1 || groups < 1) return MOE_ERR_INVALID_ARG;
  if (groups > kMxMaxGroups || static_cast<long long>(rows) * cols >= (1ll << 40)) return MOE_ERR_UNSUPPORTED;
  if (!group_offsets || !group_starts || !out || !aligned(group_offsets, 4) || !aligned(group_starts, 4) ||
      !aligned(out, 16) || (rows > 0 && (!scales || !aligned(scales, 4))))
    return MOE_ERR_INVALID_ARG;
  if (out_bytes < moe_mx_blocked_bytes(rows, cols, groups)) return MOE_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, 256) || ws_bytes < moe_mx_blocked_workspace_size(rows, groups)) return MOE_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  DeviceHeader* hdr = at<DeviceHeader*>(ws, 0);
  const size_t toff = align_up(sizeof(DeviceHeader), 256);
  const int max_tiles = rows / kGemmBM + groups;
  int32_t* tiles = at<int32_t*>(ws, toff);
  int32_t* num_tiles = at<int32_t*>(ws, toff + align_up(static_cast<size_t>(max_tiles) * 16, 256));
  cudaError_t e = launch_reset_header(hdr, s);
  if (e == cudaSuccess)
    e = launch_mx_group_blocked(scales, rows, cols, group_offsets, groups, out, group_starts, tiles, num_tiles,
                                max_tiles, hdr, s);
  return from_cuda(e);
}

moe_status moe_round_bf16(const float* y32, void* y, size_t n, moe_stream_t stream) {
  if (n == 0) return MOE_OK;
  if (!y32 || !y || !aligned(y32, 16) || !aligned(y, 16) || n % 8) return MOE_ERR_INVALID_ARG;
  return from_cuda(launch_round_bf16(y32, y, n, reinterpret_cast<cudaStream_t>(stream)));
}

moe_status moe_forward_views(const moe_problem* p, const void* ws, size_t ws_bytes, moe_views* out) {
  return moe_forward_views_ex(p, nullptr, ws, ws_bytes, out);
}

moe_status moe_forward_views_ex(const moe_problem* p, const moe_forward_options* opt, const void* ws,
                                size_t ws_bytes, moe_views* out) {
  if (!p || !out) return MOE_ERR_INVALID_ARG;
  const int S = opt ? opt->n_shared : 0;
  const moe_status vs = validate_shape(*p, S);
  if (vs != MOE_OK) return vs;
  ForwardLayout L;
  if (!plan_forward(*p, &L, S)) return MOE_ERR_UNSUPPORTED;
  if (!ws || ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  void* base = const_cast<void*>(ws);
  moe_views v{};
  v.ids = at<const int32_t*>(base, L.ids);
  v.w = at<const float*>(base, L.w);
  if (L.path == MOE_PATH_GROUPED) {
    v.counts = at<const int32_t*>(base, L.counts);
    v.offsets = at<const int32_t*>(base, L.offsets);
    v.perm = at<const int32_t*>(base, L.perm);
    v.inv = at<const int32_t*>(base, L.inv);
    v.tiles = at<const int32_t*>(base, L.tiles);
    v.num_tiles = at<const int32_t*>(base, L.num_tiles);
    if (!(p->quant == MOE_BF16 && S == 0 && gateup_gather4())) v.xs = at<const void*>(base, L.xs);
    if (p->quant == MOE_FP8_BLOCK128) v.x_scale = at<const float*>(base, L.xs_scale);
    if (p->quant == MOE_MXFP8) v.x_scale = at<const float*>(base, L.xs_sc);
  } else {
    v.xs = at<const void*>(base, L.xq);
    if (p->quant == MOE_FP8_BLOCK128) v.x_scale = at<const float*>(base, L.sx);
  }
  if (p->quant == MOE_FP8_PER_TENSOR) {
    static_assert(offsetof(DeviceHeader, amax_x) % 4 == 0, "amax_x is a 4-byte word");
    v.amax_x = reinterpret_cast<const float*>(at<const uint8_t*>(base, L.header) + offsetof(DeviceHeader, amax_x));
  }
  *out = v;
  return MOE_OK;
}

int moe_profile_start(void) { return moe_profile_start_stage(nullptr); }

int moe_profile_start_stage(const char* stage) {
  Profiler& P = prof();
  std::lock_guard<std::mutex> lk(P.mu);
  P.recycle();
  P.only = stage ? stage : "";
  P.on = true;
  return 0;
}

int moe_profile_stop(moe_stage_time* out, int max_stages) {
  Profiler& P = prof();
  std::lock_guard<std::mutex> lk(P.mu);
  P.on = false;
  std::vector<double> ms(P.names.size(), 0.0);
  std::vector<int> n(P.names.size(), 0);
  bool ok = true;
  for (const auto& r : P.records) {
    if (r.stage < 0) continue;
    if (cudaEventSynchronize(r.end) != cudaSuccess) {
      ok = false;
      continue;
    }
    float t = 0.0f;
    if (cudaEventElapsedTime(&t, r.begin, r.end) != cudaSuccess) {
      ok = false;
      continue;
    }
    ms[r.stage] += t;
    n[r.stage] += 1;
  }
  const int count = static_cast<int>(P.names.size());
  for (int i = 0; i < count && i < max_stages && out; ++i) {
    std::memset(out[i].name, 0, sizeof(out[i].name));
    std::strncpy(out[i].name, P.names[i].c_str(), sizeof(out[i].name) - 1);
    out[i].total_ms = ms[i];
    out[i].launches = n[i];
  }
  P.recycle();
  return ok ? count : -1;
}

moe_status moe_read_device_status(const void* ws, moe_stream_t stream) {
  if (!ws) return MOE_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return MOE_ERR_CUDA;
  unsigned int st = 0;
  if (cudaMemcpy(&st, ws, sizeof(st), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (st == 0) return MOE_OK;
  if (st == kStatusTimeout) return MOE_ERR_DEVICE_TIMEOUT;
  if (st == kStatusBounds) return MOE_ERR_DEVICE_BOUNDS;
  return MOE_ERR_CUDA;
}

}  // extern "C"
