// hsa_index_reindex_noalloc: the Reindex indexer for callers that must not allocate device memory.
//
// Some callers cannot create a workspace. Examples: code that runs inside a pre-planned
// memory arena owned by an inference server, plugins that may only touch the buffers they are
// handed, and latency-critical loops where an allocation (or an allocator that synchronises)
// is not acceptable. This entry point runs the same Reindex kernels as hsa_index_reindex.
// Its scratch lives in a fixed-size array in the library's own device memory, so the caller
// passes only inputs and outputs.
//
// The array below is a file-scope device symbol. Every GPU that loads the library holds it
// until the process exits. In host code its name is only a host-side stand-in, so its device
// address is looked up once per device with cudaGetSymbolAddress and passed to the kernels.
#include <string.h>

#include <mutex>

#include "hsa_common.cuh"
#include "hsa_internal.h"

namespace hsa {
namespace {

constexpr int kNoAllocMaxRows = 32;   // batch * nq
// per (request, query) row: the fused Reindex kernel's exchange areas - the lists of 64-bit
// (key, slot) composites its 4 CTAs publish (entries 0..2047 and 2048..4095 of each, in two
// regions) and their (count, valid elements) pairs
constexpr size_t kRowList = (size_t)kPool / 2 * 8;   // 4 CTAs x 2048 composites
constexpr size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }
constexpr size_t kOffListLo = 0;
constexpr size_t kOffListHi = kOffListLo + align256(kNoAllocMaxRows * kRowList);
constexpr size_t kOffCount = kOffListHi + align256(kNoAllocMaxRows * kRowList);
constexpr size_t kScratchBytes = kOffCount + align256(kNoAllocMaxRows * 2 * kRxSplit * 4);   // about 4.2 MB

static __device__ __align__(256) uint8_t g_reindex_scratch[kScratchBytes];

constexpr int kMaxDev = 64;
std::mutex g_mu;
uint8_t* g_ptr[kMaxDev];

// Device address of the scratch array on the current device (looked up once per device).
hsa_status scratch_for_current_device(uint8_t** ptr, uint32_t** status, int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return HSA_ERR_CUDA;
  if (!device_status_ptr(status, sms)) return HSA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_reindex_scratch) != cudaSuccess || !p) return HSA_ERR_CUDA;
    g_ptr[dev] = static_cast<uint8_t*>(p);
  }
  *ptr = g_ptr[dev];
  return HSA_OK;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace hsa

using namespace hsa;

extern "C" HSA_API hsa_status hsa_index_reindex_noalloc(const hsa_cache* cache, const void* q, const float* w,
                                                      const int32_t* vis, int32_t nq, int64_t max_vis,
                                                      const int32_t* pool, int32_t* topk_out, hsa_stream_t stream) {
  if (!cache || !cache->kv_q || !cache->kv_s || !cache->ik_q || !cache->ik_s) return HSA_ERR_INVALID_ARG;
  if (cache->batch < 1 || cache->capacity < 8 || (cache->capacity & 7) || cache->capacity > (int64_t)INT32_MAX)
    return HSA_ERR_SHAPE;
  if (!aligned16(cache->ik_q) || !aligned16(cache->ik_s)) return HSA_ERR_ALIGN;
  if (nq < 1 || nq > HSA_MAX_NQ || max_vis < 0 || max_vis > cache->capacity || max_vis > HSA_MAX_VIS)
    return HSA_ERR_SHAPE;
  if ((int64_t)cache->batch * nq > kNoAllocMaxRows) return HSA_ERR_SHAPE;   // beyond the fixed scratch
  if (!q || !w || !vis || !pool || !topk_out) return HSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(pool) || !aligned16(topk_out)) return HSA_ERR_ALIGN;
  uint8_t* W;
  uint32_t* status;
  int sms;
  hsa_status st = scratch_for_current_device(&W, &status, &sms);
  if (st != HSA_OK) return st;
  const cudaStream_t s = (cudaStream_t)stream;
  ReindexParams rp;
  memset(&rp, 0, sizeof(rp));
  rp.batch = cache->batch;
  rp.nq = nq;
  rp.cap = cache->capacity;
  rp.ik_q = cache->ik_q;
  rp.ik_s = cache->ik_s;
  rp.q = static_cast<const uint16_t*>(q);
  rp.w = w;
  rp.vis = vis;
  rp.pool = pool;
  rp.xlist_lo = reinterpret_cast<uint64_t*>(W + kOffListLo);
  rp.xlist_hi = reinterpret_cast<uint64_t*>(W + kOffListHi);
  rp.xcount = reinterpret_cast<int32_t*>(W + kOffCount);
  rp.ld_xcount = 2 * kRxSplit;
  rp.topk_out = topk_out;
  rp.status = status;
  if (launch_reindex(rp, s) != cudaSuccess) return HSA_ERR_CUDA;
  return HSA_OK;
}
