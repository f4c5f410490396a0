// hsa_index_full_noalloc: the Full-mode indexer for callers that cannot allocate device memory.
//
// hsa_index_full needs scratch memory between its two kernels: per-position scores, block
// maxima, histograms and candidate lists, in a workspace the caller allocates. Some callers
// cannot do that: a plugin that may only touch the buffers it is handed, code running inside a
// memory arena an inference server planned in advance, or a latency-critical loop where an
// allocator call (which may synchronise the device) is not acceptable. This entry point runs
// the same two kernels with their scratch in a fixed array that is part of the library's
// device image (kScratchBytes, 64 MiB on every device that loads the library, held until the
// process exits).
//
// Set-up: the first call on a device looks up the array's device address there
// (cudaGetSymbolAddress with that device current). In host code the array's name is only a
// host-side stand-in, so the kernels get the looked-up address. That first call should come
// before any stream capture.
//
// Every call shares the one array, which keeps whatever the last call left in it. Each call
// therefore clears the part that must start at zero (histograms and selection state) with a
// cudaMemsetAsync on its stream before the kernels run. Two calls that overlap on the GPU (on
// different streams, or from different threads) race on the array.
#include <string.h>

#include <mutex>

#include "hsa_common.cuh"
#include "hsa_internal.h"

namespace hsa {
namespace {

constexpr size_t kScratchBytes = HSA_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) uint8_t g_full_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
uint8_t* g_scratch_ptr[kMaxDevices];

// Device address of the scratch array on the current device (looked up once per device).
uint8_t* scratch_on_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_full_scratch) != cudaSuccess) return nullptr;
    g_scratch_ptr[dev] = static_cast<uint8_t*>(ptr);
  }
  return g_scratch_ptr[dev];
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace hsa

using namespace hsa;

extern "C" HSA_API hsa_status hsa_index_full_noalloc(const hsa_cache* cache, const void* q, const float* w,
                                                   const int32_t* vis, int32_t nq, int64_t max_vis,
                                                   int32_t* topk_out, int32_t* pool_out, hsa_stream_t stream) {
  hsa_status st = check_cache(cache);
  if (st != HSA_OK) return st;
  st = check_query(cache, nq, max_vis);
  if (st != HSA_OK) return st;
  if (!q || !w || !vis || !topk_out || !pool_out) return HSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(topk_out) || !aligned16(pool_out)) return HSA_ERR_ALIGN;
  WsLayout L;
  if (!make_ws_layout(cache->batch, nq, max_vis, &L)) return HSA_ERR_SHAPE;
  if (L.full_end > kScratchBytes) return HSA_ERR_WORKSPACE;   // beyond the fixed array
  uint8_t* ws = scratch_on_current_device();
  if (!ws) return HSA_ERR_CUDA;
  const cudaStream_t s = (cudaStream_t)stream;
  st = cuda_fail(cudaMemsetAsync(ws + L.zero_begin, 0, L.zero_end - L.zero_begin, s), "scratch clear");
  if (st != HSA_OK) return st;
  return launch_index_full(cache, q, w, vis, nq, max_vis, topk_out, pool_out, ws, L, s);
}
