// Host-side declarations shared by the libhsa translation units: workspace layout, kernel
// parameter blocks and launchers. Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/hsa.h"

namespace hsa {

// Workspace carve-up for hsa_index_full / hsa_index_reindex / hsa_sparse_attn_decode.
struct WsLayout {
  int32_t rows;        // batch * nq
  int64_t ld_s;        // score row stride (positions), a multiple of kScanChunk
  int64_t ld_b;        // block-max row stride (blocks) = ld_s / 8
  size_t off_scores, off_blkmax, off_hist_full, off_cand_full;
  size_t off_attn;     // attention partials
  size_t attn_bytes;
  size_t zero_begin, zero_end;   // region that must be zero between calls (the block-max histograms)
  size_t full_end;               // the Full call uses [0, full_end)
  size_t total;
};

bool make_ws_layout(int32_t batch, int32_t nq, int64_t max_vis, WsLayout* L);

// Host-side argument checks shared by the entry points (HSA_OK or the status to return).
hsa_status check_cache(const hsa_cache* c);
hsa_status check_query(const hsa_cache* c, int32_t nq, int64_t max_vis);
// Map a CUDA error to HSA_ERR_CUDA; with HSA_DEBUG set in the environment, name it on stderr.
hsa_status cuda_fail(cudaError_t e, const char* where);

// The Full-mode indexer (scan, then selection) over checked arguments, with its scratch regions
// at `ws` laid out by L. The region [L.zero_begin, L.zero_end) must be zero on entry; the
// kernels leave it zero.
hsa_status launch_index_full(const hsa_cache* cache, const void* q, const float* w, const int32_t* vis, int32_t nq,
                             int64_t max_vis, int32_t* topk_out, int32_t* pool_out, uint8_t* ws,
                             const WsLayout& L, cudaStream_t s);

// Device address of the per-device status word and the SM count of the current device;
// false on a non-sm_100-family device.
bool device_status_ptr(uint32_t** status, int* sms);

// Limit of the kernels' bounded waits for the next launches (hsa_set_wait_limit), in ns.
uint64_t wait_limit_ns();

// Raise the dynamic shared-memory limit of kernel `func` to `bytes` on the current device. The
// attribute belongs to the device's context, so it is set once per (device, kernel) and again
// whenever a larger size is asked for; thread-safe.
cudaError_t ensure_smem_limit(const void* func, size_t bytes);

// ------------------------------------------------------------------ index scoring
struct ScanParams {         // Full mode: a segment is one request, its nq queries share K
  int32_t batch, nq;
  int64_t cap;
  const uint8_t* ik_q;
  const uint8_t* ik_s;
  const uint16_t* q;     // bf16 [B][nq][16][128]
  const float* w;        // [B][nq][16]
  const int32_t* vis;    // [B][nq]
  int32_t n_seg;
  int32_t chunks_per_seg;
  int32_t total_items;
  float* scores;         // [rows][ld_s]
  int64_t ld_s;
  float* blkmax;         // [rows][ld_b]
  int64_t ld_b;
  uint32_t* hist;        // [rows][4096] counts of the block maxima's top 12 key bits
  uint32_t* status;
  uint64_t wait_ns;      // bounded-wait limit
  int32_t stall_last;    // test hook: CTA 0's producer withholds the copy of its last stage
};

struct SelectParams {       // the Full step's block top-2048 (pool) and position top-512
  int32_t batch, nq;
  int64_t max_vis;
  const int32_t* vis;
  const float* scores;
  int64_t ld_s;
  const float* blkmax;
  int64_t ld_b;
  uint32_t* hist;        // [rows][4096], cleared by the selection
  int32_t* cand;         // [rows][2 * ld_b] threshold-bin candidates past the shared-memory stage
  int64_t ld_cand;
  int32_t* topk_out;     // [rows][512]
  int32_t* pool_out;     // [rows][pool_ld]
  int64_t pool_ld;       // 16384, or 16384 + 160 with the window tail
  int32_t tail;          // 1: the window's blocks join the pool
  uint32_t* status;
};

cudaError_t launch_index_scan(const ScanParams& p, int num_sms, cudaStream_t s);
cudaError_t launch_select(const SelectParams& p, cudaStream_t s);

// ------------------------------------------------------------------ fused Reindex (one cluster per row)
struct ReindexParams {
  int32_t batch, nq;
  int64_t cap;
  const uint8_t* ik_q;
  const uint8_t* ik_s;
  const uint16_t* q;     // bf16 [B][nq][16][128]
  const float* w;        // [B][nq][16]
  const int32_t* vis;    // [B][nq]
  const int32_t* pool;   // [B][nq][pool_ld]
  int64_t pool_ld;       // 16384, or 16384 + 160 with the window tail
  int32_t tail;          // 1: CTA rank 3 also scores the 160 slots past 16384
  int32_t* topk_out;     // [B][nq][512]
  uint32_t* status;
  int32_t inputs_ready;  // 1: q, w, vis and pool are complete at launch (schedule_step); the kernel then waits
                         // on the previous kernel only before its first global write
};
cudaError_t launch_reindex(const ReindexParams& p, cudaStream_t s);

// ------------------------------------------------------------------ attention
struct AttnParams {
  CUtensorMap qmap;       // q as a 2-D bf16 tensor [B*nq*64][512], 64 x 16 boxes, 128-byte swizzle
  int32_t batch, nq;
  int64_t cap;
  int32_t scale_fmt;
  const uint8_t* kv_q;
  const uint8_t* kv_s;
  const uint16_t* q;      // bf16 [B][nq][64][512]
  const int32_t* topk;    // [B][nq][512]
  const uint8_t* swa;     // [B][W+nq-1][512]
  const int32_t* vis;     // [B][nq]
  float sm_scale;
  int32_t inputs_ready;   // 1: q and swa are complete at launch (schedule_step), read before the dependency wait
  int32_t topk_ready;     // 1 (with inputs_ready): topk is two or more kernels old (a Reuse slot); the kernel
                          // waits for the previous one only before its first global write
  float* out;             // [B][nq][64][512]
  float* partial;         // workspace: [B*nq][4][64*512 outputs, then 64 (max, sum) pairs]
  uint32_t* status;
  uint64_t wait_ns;       // bounded-wait limit
};
cudaError_t launch_attention(const AttnParams& p, cudaStream_t s);

// ------------------------------------------------------------------ cache write
struct WriteParams {
  int32_t batch, ratio, scale_fmt;
  int64_t cap, n_tokens, n_entries;
  const uint16_t* wkv;
  const uint16_t* wgate;
  const uint16_t* w_idx;
  const int64_t* start_entry;
  uint8_t* kv_q;
  uint8_t* kv_s;
  uint8_t* ik_q;
  uint8_t* ik_s;
  uint32_t* status;
  uint64_t wait_ns;                          // bounded-wait limit
  int32_t rope;                              // 1: rotate the main-KV latent's last 64 dims
  uint64_t rope_turns[HSA_ROPE_DIMS / 2];    // turns per position of pair k, a 64-bit binary fraction
};
cudaError_t launch_cache_write(const WriteParams& p, cudaStream_t s);

}  // namespace hsa
