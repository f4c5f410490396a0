// C ABI of libhsa (include/hsa.h): argument validation, workspace carve-up, launches and the
// decode-step schedule. Everything here is host code; it launches kernels only.
#include <math.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include <nvtx3/nvToolsExt.h>

#include "hsa_common.cuh"
#include "hsa_internal.h"

namespace hsa {

// NVTX range of one C-ABI call (or one layer slot of a step) in the "libhsa" domain, so that a
// timeline tool attributes the call's host time and its launches; costs a pointer test when no
// tool is attached.
class NvtxRange {
 public:
  explicit NvtxRange(const char* name) {
    static const nvtxDomainHandle_t domain = nvtxDomainCreateA("libhsa");
    nvtxEventAttributes_t a = {};
    a.version = NVTX_VERSION;
    a.size = NVTX_EVENT_ATTRIB_STRUCT_SIZE;
    a.messageType = NVTX_MESSAGE_TYPE_ASCII;
    a.message.ascii = name;
    domain_ = domain;
    nvtxDomainRangePushEx(domain_, &a);
  }
  ~NvtxRange() { nvtxDomainRangePop(domain_); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;

 private:
  nvtxDomainHandle_t domain_;
};

// Per-device status word (HSA_FLAG_*), written by kernels with atomicOr.
__device__ uint32_t g_status_word;

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
uint32_t* g_status_ptr[kMaxDevices];
int g_num_sms[kMaxDevices];
int g_cc_major[kMaxDevices];

// Device pointer of the status word and the SM count of the current device (set up once per device).
bool device_info(uint32_t** status, int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_status_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_status_word) != cudaSuccess) return false;
    cudaDeviceGetAttribute(&g_num_sms[dev], cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&g_cc_major[dev], cudaDevAttrComputeCapabilityMajor, dev);
    g_status_ptr[dev] = static_cast<uint32_t*>(ptr);
  }
  *status = g_status_ptr[dev];
  *sms = g_num_sms[dev];
  return g_cc_major[dev] == 10;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

}  // namespace

hsa_status cuda_fail(cudaError_t e, const char* where) {
  if (e == cudaSuccess) return HSA_OK;
  static const bool dbg = getenv("HSA_DEBUG") != nullptr;
  if (dbg) fprintf(stderr, "hsa: %s: %s\n", where, cudaGetErrorString(e));
  return HSA_ERR_CUDA;
}

hsa_status check_cache(const hsa_cache* c) {
  if (!c || !c->kv_q || !c->kv_s || !c->ik_q || !c->ik_s) return HSA_ERR_INVALID_ARG;
  if (c->batch < 1 || c->capacity < 8 || (c->capacity & 7)) return HSA_ERR_SHAPE;
  if (c->capacity > (int64_t)INT32_MAX) return HSA_ERR_SHAPE;
  if (c->ratio != 1 && c->ratio != 2) return HSA_ERR_INVALID_ARG;
  if (c->kv_scale_fmt != HSA_SCALE_E8M0 && c->kv_scale_fmt != HSA_SCALE_E4M3) return HSA_ERR_INVALID_ARG;
  if ((uint32_t)c->flags & ~(HSA_CACHE_ROPE | HSA_CACHE_POOL_TAIL)) return HSA_ERR_INVALID_ARG;
  if (!aligned16(c->kv_q) || !aligned16(c->kv_s) || !aligned16(c->ik_q) || !aligned16(c->ik_s)) return HSA_ERR_ALIGN;
  return HSA_OK;
}

hsa_status check_query(const hsa_cache* c, int32_t nq, int64_t max_vis) {
  if (nq < 1 || nq > HSA_MAX_NQ) return HSA_ERR_SHAPE;
  if (max_vis < 0 || max_vis > c->capacity || max_vis > HSA_MAX_VIS) return HSA_ERR_SHAPE;
  return HSA_OK;
}

bool device_status_ptr(uint32_t** status, int* sms) { return device_info(status, sms); }

namespace {
std::atomic<uint64_t> g_wait_ns{kWaitLimitNs};   // bounded-wait limit of the next launches
std::atomic<int> g_stall_next_scan{0};           // test hook, consumed by the next Full call
}  // namespace

uint64_t wait_limit_ns() { return g_wait_ns.load(std::memory_order_relaxed); }

namespace {
struct SmemLimit {
  int dev;
  const void* func;
  size_t bytes;
};
constexpr int kMaxSmemLimits = 256;
SmemLimit g_smem_limits[kMaxSmemLimits];
int g_n_smem_limits = 0;
}  // namespace

cudaError_t ensure_smem_limit(const void* func, size_t bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(g_mu);
  int slot = -1;
  for (int i = 0; i < g_n_smem_limits; ++i)
    if (g_smem_limits[i].dev == dev && g_smem_limits[i].func == func) slot = i;
  if (slot >= 0 && g_smem_limits[slot].bytes >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  if (slot < 0) {
    if (g_n_smem_limits == kMaxSmemLimits) return cudaSuccess;   // set on every call from here on
    slot = g_n_smem_limits++;
    g_smem_limits[slot].dev = dev;
    g_smem_limits[slot].func = func;
  }
  g_smem_limits[slot].bytes = bytes;
  return cudaSuccess;
}

bool make_ws_layout(int32_t batch, int32_t nq, int64_t max_vis, WsLayout* L) {
  if (batch < 1 || nq < 1 || nq > HSA_MAX_NQ || max_vis < 0 || max_vis > HSA_MAX_VIS) return false;
  const int64_t rows = (int64_t)batch * nq;
  L->rows = (int32_t)rows;
  L->ld_s = round_up(std::max(max_vis, (int64_t)1), kScanChunk);
  L->ld_b = L->ld_s / 8;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o += (bytes + 255) & ~(size_t)255;
    return at;
  };
  // zero-between-calls region first: the block-max histograms of the Full scan
  L->zero_begin = 0;
  L->off_hist_full = take((size_t)rows * kHistBins * 4);
  L->zero_end = o;
  L->off_scores = take((size_t)rows * L->ld_s * 4);
  L->off_blkmax = take((size_t)rows * L->ld_b * 4);
  L->off_cand_full = take((size_t)rows * 2 * L->ld_b * 4);
  L->full_end = o;
  // attention partials: per row, 4 CTAs x (64 x 512 unnormalised outputs + 64 (max, sum) pairs)
  L->attn_bytes = (size_t)rows * kAttnSplit * (kHAtt * kDLat + 2 * kHAtt) * 4;
  L->off_attn = take(L->attn_bytes);
  L->total = o;
  return true;
}

hsa_status launch_index_full(const hsa_cache* cache, const void* q, const float* w, const int32_t* vis, int32_t nq,
                             int64_t max_vis, int32_t* topk_out, int32_t* pool_out, uint8_t* W,
                             const WsLayout& L, cudaStream_t s) {
  uint32_t* status;
  int sms;
  if (!device_info(&status, &sms)) return HSA_ERR_UNSUPPORTED;
  ScanParams sp;
  memset(&sp, 0, sizeof(sp));
  sp.batch = cache->batch;
  sp.nq = nq;
  sp.cap = cache->capacity;
  sp.ik_q = cache->ik_q;
  sp.ik_s = cache->ik_s;
  sp.q = static_cast<const uint16_t*>(q);
  sp.w = w;
  sp.vis = vis;
  sp.status = status;
  sp.n_seg = cache->batch;
  sp.chunks_per_seg = (int32_t)((std::max(max_vis, (int64_t)1) + kScanChunk - 1) / kScanChunk);
  sp.total_items = sp.n_seg * sp.chunks_per_seg;
  sp.scores = reinterpret_cast<float*>(W + L.off_scores);
  sp.ld_s = L.ld_s;
  sp.blkmax = reinterpret_cast<float*>(W + L.off_blkmax);
  sp.ld_b = L.ld_b;
  sp.hist = reinterpret_cast<uint32_t*>(W + L.off_hist_full);
  sp.wait_ns = wait_limit_ns();
  sp.stall_last = g_stall_next_scan.exchange(0);
  SelectParams se;
  memset(&se, 0, sizeof(se));
  se.batch = cache->batch;
  se.nq = nq;
  se.max_vis = max_vis;
  se.vis = vis;
  se.topk_out = topk_out;
  se.pool_out = pool_out;
  se.status = status;
  se.scores = sp.scores;
  se.ld_s = sp.ld_s;
  se.blkmax = sp.blkmax;
  se.ld_b = sp.ld_b;
  se.hist = sp.hist;
  se.cand = reinterpret_cast<int32_t*>(W + L.off_cand_full);
  se.ld_cand = 2 * L.ld_b;
  se.tail = (cache->flags & HSA_CACHE_POOL_TAIL) ? 1 : 0;
  se.pool_ld = kPool + (se.tail ? HSA_POOL_TAIL_SLOTS : 0);
  hsa_status r = cuda_fail(launch_index_scan(sp, sms, s), "index scan launch");
  if (r != HSA_OK) return r;
  return cuda_fail(launch_select(se, s), "select launch");
}

// inputs_ready: q and swa are complete when the kernel is launched (no kernel of the same
// schedule_step writes them), so the kernel may fetch them before its programmatic-dependency
// wait; topk_ready: topk was written two or more kernels earlier (a Reuse slot), so the kernel
// waits only before its first global write.
hsa_status attn_common(const hsa_cache* cache, const void* q, const int32_t* topk, const uint8_t* swa,
                       const int32_t* vis, int32_t nq, int64_t max_vis, float sm_scale, float* out, void* ws,
                       size_t ws_bytes, hsa_stream_t stream, bool inputs_ready, bool topk_ready) {
  hsa_status st = check_cache(cache);
  if (st != HSA_OK) return st;
  st = check_query(cache, nq, max_vis);
  if (st != HSA_OK) return st;
  if (!q || !topk || !swa || !vis || !out) return HSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(swa) || !aligned16(out)) return HSA_ERR_ALIGN;
  WsLayout L;
  if (!make_ws_layout(cache->batch, nq, max_vis, &L)) return HSA_ERR_SHAPE;
  if (!ws || ws_bytes < L.total) return HSA_ERR_WORKSPACE;
  if (!aligned16(ws)) return HSA_ERR_ALIGN;
  uint32_t* status;
  int sms;
  if (!device_info(&status, &sms)) return HSA_ERR_UNSUPPORTED;
  AttnParams p;
  memset(&p, 0, sizeof(p));
  p.batch = cache->batch;
  p.nq = nq;
  p.cap = cache->capacity;
  p.scale_fmt = cache->kv_scale_fmt;
  p.kv_q = cache->kv_q;
  p.kv_s = cache->kv_s;
  p.q = static_cast<const uint16_t*>(q);
  p.topk = topk;
  p.swa = swa;
  p.vis = vis;
  p.sm_scale = sm_scale;
  p.inputs_ready = inputs_ready ? 1 : 0;
  p.topk_ready = (inputs_ready && topk_ready) ? 1 : 0;
  p.out = out;
  p.partial = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + L.off_attn);
  p.status = status;
  p.wait_ns = wait_limit_ns();
  return cuda_fail(launch_attention(p, (cudaStream_t)stream), "attention launch");
}
}  // namespace hsa

using namespace hsa;

extern "C" {

int32_t hsa_abi_version(void) { return HSA_ABI_VERSION; }

const char* hsa_status_string(hsa_status s) {
  switch (s) {
    case HSA_OK: return "HSA_OK";
    case HSA_ERR_INVALID_ARG: return "HSA_ERR_INVALID_ARG: a pointer is NULL or an enum/size is invalid";
    case HSA_ERR_SHAPE: return "HSA_ERR_SHAPE: a size is out of range";
    case HSA_ERR_ALIGN: return "HSA_ERR_ALIGN: a pointer is not 16-byte aligned";
    case HSA_ERR_WORKSPACE: return "HSA_ERR_WORKSPACE: workspace missing or too small";
    case HSA_ERR_CUDA: return "HSA_ERR_CUDA: a CUDA call or kernel launch failed";
    case HSA_ERR_TIMEOUT: return "HSA_ERR_TIMEOUT: a bounded device wait gave up";
    case HSA_ERR_UNSUPPORTED: return "HSA_ERR_UNSUPPORTED: needs an sm_100-family GPU (GB300 / sm_103a)";
  }
  return "HSA_ERR_UNKNOWN";
}

size_t hsa_workspace_bytes(int32_t batch, int32_t nq, int64_t max_vis) {
  WsLayout L;
  if (!make_ws_layout(batch, nq, max_vis, &L)) return 0;
  return L.total;
}

hsa_status hsa_workspace_init(void* ws, size_t ws_bytes, hsa_stream_t stream) {
  if (!ws) return HSA_ERR_INVALID_ARG;
  return cudaMemsetAsync(ws, 0, ws_bytes, (cudaStream_t)stream) == cudaSuccess ? HSA_OK : HSA_ERR_CUDA;
}

hsa_status hsa_cache_write_compress(const hsa_cache* cache, const void* wkv, const void* wgate, const void* w_idx,
                                    int64_t n_tokens, const int64_t* start_entry, hsa_stream_t stream) {
  NvtxRange range("hsa_cache_write_compress");
  hsa_status st = check_cache(cache);
  if (st != HSA_OK) return st;
  if (!wkv || !w_idx) return HSA_ERR_INVALID_ARG;
  if ((cache->ratio == 2) != (wgate != nullptr)) return HSA_ERR_INVALID_ARG;
  if (n_tokens < 0) return HSA_ERR_SHAPE;
  if (!aligned16(wkv) || !aligned16(w_idx) || (wgate && !aligned16(wgate))) return HSA_ERR_ALIGN;
  uint32_t* status;
  int sms;
  if (!device_info(&status, &sms)) return HSA_ERR_UNSUPPORTED;
  WriteParams p;
  memset(&p, 0, sizeof(p));
  p.batch = cache->batch;
  p.ratio = cache->ratio;
  p.scale_fmt = cache->kv_scale_fmt;
  p.cap = cache->capacity;
  p.n_tokens = n_tokens;
  p.n_entries = n_tokens / cache->ratio;
  p.wkv = static_cast<const uint16_t*>(wkv);
  p.wgate = static_cast<const uint16_t*>(wgate);
  p.w_idx = static_cast<const uint16_t*>(w_idx);
  p.start_entry = start_entry;
  p.kv_q = cache->kv_q;
  p.kv_s = cache->kv_s;
  p.ik_q = cache->ik_q;
  p.ik_s = cache->ik_s;
  p.status = status;
  p.wait_ns = wait_limit_ns();
  if (cache->flags & HSA_CACHE_ROPE) {
    // RoPE turns per position of pair k, theta^(-k/32) / 2 pi, as a 64-bit binary fraction: the
    // phase of entry e is then the wrapping product e * turns (mod one turn, exactly)
    p.rope = 1;
    for (int k = 0; k < HSA_ROPE_DIMS / 2; ++k) {
      const double f = pow(HSA_ROPE_THETA, -2.0 * k / HSA_ROPE_DIMS) / (2.0 * 3.14159265358979323846);
      p.rope_turns[k] = (uint64_t)ldexp(f, 64);
    }
  }
  if (p.n_entries == 0) return HSA_OK;
  return cuda_fail(launch_cache_write(p, (cudaStream_t)stream), "cache write launch");
}

static hsa_status index_common(bool pool_mode, const hsa_cache* cache, const void* q, const float* w,
                               const int32_t* vis, int32_t nq, int64_t max_vis, const int32_t* pool,
                               int32_t* topk_out, int32_t* pool_out, void* ws, size_t ws_bytes,
                               hsa_stream_t stream, bool inputs_ready = false) {
  hsa_status st = check_cache(cache);
  if (st != HSA_OK) return st;
  st = check_query(cache, nq, max_vis);
  if (st != HSA_OK) return st;
  if (!q || !w || !vis || !topk_out || (pool_mode ? !pool : !pool_out)) return HSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(topk_out) || (pool_out && !aligned16(pool_out)) || (pool && !aligned16(pool)))
    return HSA_ERR_ALIGN;
  WsLayout L;
  if (!make_ws_layout(cache->batch, nq, max_vis, &L)) return HSA_ERR_SHAPE;
  if (!ws || ws_bytes < L.total) return HSA_ERR_WORKSPACE;
  if (!aligned16(ws)) return HSA_ERR_ALIGN;
  uint32_t* status;
  int sms;
  if (!device_info(&status, &sms)) return HSA_ERR_UNSUPPORTED;
  uint8_t* W = static_cast<uint8_t*>(ws);
  const cudaStream_t s = (cudaStream_t)stream;

  if (pool_mode) {
    // one fused launch: rescoring over the pool and the exact top-512, one cluster per row; its
    // CTAs exchange their candidate lists through distributed shared memory, so the workspace
    // is not touched
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
    rp.tail = (cache->flags & HSA_CACHE_POOL_TAIL) ? 1 : 0;
    rp.pool_ld = kPool + (rp.tail ? HSA_POOL_TAIL_SLOTS : 0);
    rp.topk_out = topk_out;
    rp.status = status;
    rp.inputs_ready = inputs_ready ? 1 : 0;
    return cuda_fail(launch_reindex(rp, s), "reindex launch");
  }

  return launch_index_full(cache, q, w, vis, nq, max_vis, topk_out, pool_out, W, L, s);
}

hsa_status hsa_index_full(const hsa_cache* cache, const void* q, const float* w, const int32_t* vis, int32_t nq,
                          int64_t max_vis, int32_t* topk_out, int32_t* pool_out, void* ws, size_t ws_bytes,
                          hsa_stream_t stream) {
  NvtxRange range("hsa_index_full");
  return index_common(false, cache, q, w, vis, nq, max_vis, nullptr, topk_out, pool_out, ws, ws_bytes, stream);
}

hsa_status hsa_index_reindex(const hsa_cache* cache, const void* q, const float* w, const int32_t* vis, int32_t nq,
                             int64_t max_vis, const int32_t* pool, int32_t* topk_out, void* ws, size_t ws_bytes,
                             hsa_stream_t stream) {
  NvtxRange range("hsa_index_reindex");
  return index_common(true, cache, q, w, vis, nq, max_vis, pool, topk_out, nullptr, ws, ws_bytes, stream);
}


hsa_status hsa_sparse_attn_decode(const hsa_cache* cache, const void* q, const int32_t* topk, const uint8_t* swa,
                                  const int32_t* vis, int32_t nq, int64_t max_vis, float sm_scale, float* out,
                                  void* ws, size_t ws_bytes, hsa_stream_t stream) {
  NvtxRange range("hsa_sparse_attn_decode");
  return attn_common(cache, q, topk, swa, vis, nq, max_vis, sm_scale, out, ws, ws_bytes, stream, false, false);
}

hsa_status hsa_schedule_step(const hsa_cache* caches, const hsa_step_args* a, void* ws, size_t ws_bytes,
                             hsa_stream_t stream) {
  NvtxRange range("hsa_schedule_step");
  if (!caches || !a || !a->modes || !a->q_attn || !a->swa || !a->out || !a->topk || !a->pool || !a->vis)
    return HSA_ERR_INVALID_ARG;
  if (a->n_layers < 1) return HSA_ERR_SHAPE;
  if (a->modes[0] != HSA_MODE_FULL) return HSA_ERR_INVALID_ARG;
  // every slot's cache is checked before anything is launched; the pool's row length follows
  // the pool-tail flag, so all slots must agree on it
  for (int l = 0; l < a->n_layers; ++l) {
    const hsa_status cs = check_cache(caches + l);
    if (cs != HSA_OK) return cs;
    if (caches[l].batch != caches[0].batch || caches[l].ratio != caches[0].ratio ||
        ((caches[l].flags ^ caches[0].flags) & HSA_CACHE_POOL_TAIL) || a->max_vis > caches[l].capacity)
      return HSA_ERR_SHAPE;
  }
  hsa_status st = HSA_OK;
  for (int l = 0; l < a->n_layers; ++l) {
    const int m = a->modes[l];
    if (m != HSA_MODE_FULL && m != HSA_MODE_REINDEX && m != HSA_MODE_REUSE) return HSA_ERR_INVALID_ARG;
    if (m != HSA_MODE_REUSE && (!a->q_idx || !a->w_idx || !a->q_idx[l] || !a->w_idx[l] || !a->topk[l]))
      return HSA_ERR_INVALID_ARG;
    if (!a->q_attn[l] || !a->swa[l] || !a->out[l]) return HSA_ERR_INVALID_ARG;
  }
  const int32_t* latest = nullptr;
  static const char* const kSlotName[3] = {"layer slot: Full + attention", "layer slot: Reindex + attention",
                                           "layer slot: Reuse + attention"};
  for (int l = 0; l < a->n_layers; ++l) {
    const int m = a->modes[l];
    NvtxRange slot(kSlotName[m]);
    const hsa_cache* cache = caches + l;
    if (m == HSA_MODE_FULL) {
      st = hsa_index_full(cache, a->q_idx[l], a->w_idx[l], a->vis, a->nq, a->max_vis, a->topk[l], a->pool, ws,
                          ws_bytes, stream);
      latest = a->topk[l];
    } else if (m == HSA_MODE_REINDEX) {
      // the pool was written at least two kernels earlier and q_idx, w_idx are step inputs: the
      // kernel may read them before its programmatic-dependency wait
      st = index_common(true, cache, a->q_idx[l], a->w_idx[l], a->vis, a->nq, a->max_vis, a->pool, a->topk[l],
                        nullptr, ws, ws_bytes, stream, true);
      latest = a->topk[l];
    }
    if (st != HSA_OK) return st;
    st = attn_common(cache, a->q_attn[l], latest, a->swa[l], a->vis, a->nq, a->max_vis, a->sm_scale,
                                a->out[l], ws, ws_bytes, stream, true, m == HSA_MODE_REUSE);
    if (st != HSA_OK) return st;
  }
  return HSA_OK;
}

hsa_status hsa_set_wait_limit(uint64_t ns) {
  g_wait_ns.store(ns ? ns : kWaitLimitNs, std::memory_order_relaxed);
  return HSA_OK;
}

hsa_status hsa_debug_stall_next_scan(void) {
  g_stall_next_scan.store(1);
  return HSA_OK;
}

hsa_status hsa_get_device_status(hsa_stream_t stream, uint32_t* flags) {
  if (!flags) return HSA_ERR_INVALID_ARG;
  uint32_t* status;
  int sms;
  device_info(&status, &sms);
  if (!status) return HSA_ERR_CUDA;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return HSA_ERR_CUDA;
  uint32_t v = 0;
  if (cudaMemcpy(&v, status, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return HSA_ERR_CUDA;
  if (cudaMemset(status, 0, 4) != cudaSuccess) return HSA_ERR_CUDA;
  *flags = v;
  return (v & HSA_FLAG_TIMEOUT) ? HSA_ERR_TIMEOUT : HSA_OK;
}

}  // extern "C"
