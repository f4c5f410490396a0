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
// per (request, query) row: slot scores, candidates, sure list, histogram, select state, done flag
constexpr size_t kRowHist = (size_t)kHistBins * 4;
constexpr size_t kRowScores = (size_t)kPool * 4;
constexpr size_t kRowCand = (size_t)kPool * 4;
constexpr size_t kRowSure = (size_t)kTopK * 4;
constexpr size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }
constexpr size_t kOffHist = 0;
constexpr size_t kOffState = kOffHist + align256(kNoAllocMaxRows * kRowHist);
constexpr size_t kOffDone = kOffState + align256(kNoAllocMaxRows * sizeof(SelState));
constexpr size_t kZeroEnd = kOffDone + align256(kNoAllocMaxRows * 4);
constexpr size_t kOffScores = kZeroEnd;
constexpr size_t kOffCand = kOffScores + align256(kNoAllocMaxRows * kRowScores);
constexpr size_t kOffSure = kOffCand + align256(kNoAllocMaxRows * kRowCand);
constexpr size_t kScratchBytes = kOffSure + align256(kNoAllocMaxRows * kRowSure);   // about 4.7 MB

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
  const int32_t rows = cache->batch * nq;
  // the histogram / select-state / done-flag region must start at zero
  if (cudaMemsetAsync(W, 0, kZeroEnd, s) != cudaSuccess) return HSA_ERR_CUDA;

  ScanParams sp;
  memset(&sp, 0, sizeof(sp));
  sp.pool_mode = 1;
  sp.batch = cache->batch;
  sp.nq = nq;
  sp.cap = cache->capacity;
  sp.ik_q = cache->ik_q;
  sp.ik_s = cache->ik_s;
  sp.q = static_cast<const uint16_t*>(q);
  sp.w = w;
  sp.vis = vis;
  sp.pool = pool;
  sp.n_seg = rows;
  sp.chunks_per_seg = kPool / kScanChunk;
  sp.total_items = sp.n_seg * sp.chunks_per_seg;
  sp.scores = reinterpret_cast<float*>(W + kOffScores);
  sp.ld_s = kPool;
  sp.hist = reinterpret_cast<uint32_t*>(W + kOffHist);
  sp.state = reinterpret_cast<SelState*>(W + kOffState);
  sp.seg_done = reinterpret_cast<uint32_t*>(W + kOffDone);
  sp.status = status;

  SelectParams se;
  memset(&se, 0, sizeof(se));
  se.pool_mode = 1;
  se.batch = cache->batch;
  se.nq = nq;
  se.max_vis = max_vis;
  se.vis = vis;
  se.pool = pool;
  se.scores = sp.scores;
  se.ld_s = kPool;
  se.hist = sp.hist;
  se.state = sp.state;
  se.cand = reinterpret_cast<int32_t*>(W + kOffCand);
  se.ld_cand = kPool;
  se.sure = reinterpret_cast<int32_t*>(W + kOffSure);
  se.ld_sure = kTopK;
  se.topk_out = topk_out;
  se.status = status;
  if (launch_index_scan(sp, sms, s) != cudaSuccess) return HSA_ERR_CUDA;
  if (launch_select(se, s) != cudaSuccess) return HSA_ERR_CUDA;
  return HSA_OK;
}
