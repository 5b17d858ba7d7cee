// moe_shuffle_noalloc: the index shuffle for callers that cannot allocate.
//
// Some callers cannot obtain device memory at the moment they need the shuffle:
// code that runs while a stream is being captured into a CUDA graph (cudaMalloc
// is not allowed during capture), plugins run by a host framework that owns all
// device memory and hands out no scratch buffer, and serving loops that forbid
// allocation after start-up so that their memory footprint stays fixed.  This
// entry point serves them: it runs the same kernels as moe_shuffle, but its
// scratch lives in a fixed array compiled into the library, so neither the caller
// nor the library allocates anything.  The caller still passes the inputs and the
// outputs.
//
// The array is a static __device__ object: every GPU on which the library is
// loaded holds its kNoallocScratchBytes from module load until the process exits.
// Its name, used in host code, is only a host-side stand-in for the symbol, never
// a device address, so the device address is looked up with
// cudaGetSymbolAddress() on the first call on each device (with that device
// current) and cached; that first call should therefore happen before any stream
// capture begins.  All calls share the one array and it keeps whatever the last
// call left in it: the status header is cleared at the start of every call and
// every other scratch word is fully written before it is read.  Calls whose work
// overlaps on the GPU (for example on two streams at once) race on the array and
// must be serialised by the caller.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr size_t kNoallocScratchBytes = MOE_NOALLOC_SCRATCH_BYTES;
static_assert(kNoallocScratchBytes % 256 == 0, "scratch is a whole number of 256-byte blocks");

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device (looked up once per device).
cudaError_t noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    if (!p) return cudaErrorInvalidSymbol;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status moe_shuffle_noalloc(const int32_t* ids, int T, int E, int k, int32_t* counts,
                                          int32_t* offsets, int32_t* perm, int32_t* inv, moe_stream_t stream) {
  if (T < 0 || E < 1 || k < 1 || k > E) return MOE_ERR_INVALID_ARG;
  if (E > kMaxE || k > kMaxK || static_cast<long long>(T) * k >= (1ll << 31)) return MOE_ERR_UNSUPPORTED;
  if (!counts || !offsets || reinterpret_cast<uintptr_t>(counts) % 4 || reinterpret_cast<uintptr_t>(offsets) % 4)
    return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!ids || !perm || !inv || reinterpret_cast<uintptr_t>(ids) % 4 ||
                reinterpret_cast<uintptr_t>(perm) % 4 || reinterpret_cast<uintptr_t>(inv) % 4))
    return MOE_ERR_INVALID_ARG;
  // the problem's scratch must fit the fixed array
  const ShuffleLayout L = plan_shuffle(T, E, k, align_up(sizeof(DeviceHeader), 256));
  if (L.total > kNoallocScratchBytes) return MOE_ERR_WORKSPACE;

  void* ws = nullptr;
  if (noalloc_scratch(&ws) != cudaSuccess) return MOE_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  DeviceHeader* hdr = reinterpret_cast<DeviceHeader*>(ws);
  cudaError_t e = launch_reset_header(hdr, s);
  if (e == cudaSuccess && T == 0) {
    e = cudaMemsetAsync(counts, 0, static_cast<size_t>(E) * 4, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(offsets, 0, static_cast<size_t>(E + 1) * 4, s);
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
  }
  int32_t* lrank = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) + L.lrank);
  int32_t* bc = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) + L.blockcounts);
  if (e == cudaSuccess)
    e = launch_route_rank(nullptr, ids, T, E, k, nullptr, nullptr, lrank, bc, hdr, false, true, s);
  if (e == cudaSuccess)
    e = launch_scan_tiles(bc, L.nblk, E, counts, offsets, nullptr, nullptr, 0, kGemmBM, nullptr, hdr, s);
  if (e == cudaSuccess) e = launch_scatter(ids, lrank, bc, T, E, k, perm, inv, s);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
