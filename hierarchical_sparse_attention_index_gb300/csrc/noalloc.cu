// hsa_index_reindex_noalloc: the Reindex indexer for callers that must not allocate device memory.
//
// Some callers cannot create a workspace. Examples: code that runs inside a pre-planned
// memory arena owned by an inference server, plugins that may only touch the buffers they are
// handed, and latency-critical loops where an allocation (or an allocator that synchronises)
// is not acceptable. This entry point runs the same fused Reindex kernel as hsa_index_reindex.
// That kernel keeps everything it exchanges between the CTAs of a row in shared memory, so the
// caller passes only inputs and outputs and no scratch memory is involved.
#include <string.h>

#include "hsa_common.cuh"
#include "hsa_internal.h"

namespace hsa {
namespace {
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
  if (!q || !w || !vis || !pool || !topk_out) return HSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(pool) || !aligned16(topk_out)) return HSA_ERR_ALIGN;
  uint32_t* status;
  int sms;
  if (!device_status_ptr(&status, &sms)) return HSA_ERR_UNSUPPORTED;
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
  rp.topk_out = topk_out;
  rp.status = status;
  if (launch_reindex(rp, (cudaStream_t)stream) != cudaSuccess) return HSA_ERR_CUDA;
  return HSA_OK;
}
