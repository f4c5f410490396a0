/*
 * hsa.h — C ABI of libhsa: the decode-time CSA2 hierarchical sparse indexer, the sparse
 * attention over FP4 main KV + FP8 SWA tail, and the compressed-cache write of
 * DeepSeek-V4.1-Flash, as hand-written CUDA kernels for GB300 (sm_103a).
 *
 * Sources. The pages are cited by tag, title and section:
 *   [890B]  jokeuncle.pages.dev, "两张架构图里藏着 890 字节：把 DeepSeek V4.1 Flash 的 43 层排班表算出来"
 *   [COST]  weigao.cc, "DeepSeek V4.1 Flash：从架构到推理成本"
 *   [CED]   syt-nju.github.io, "DeepSeek-V4.1-Flash：为什么读输入只激活 8B，写输出要 16B"
 *   [ARCH]  ggaaooppeenngg.github.io, "DeepSeek-V4.1-Flash 架构解析：KV Cache 压缩的极限在哪里"
 *   [10100] 10100.com, DeepSeek-V4.1-Flash Architecture, 层次化稀疏索引器
 *
 * Conventions shared by every call:
 *  - All pointers in argument lists are DEVICE pointers unless marked "host". They are owned
 *    by the caller. The library never allocates, frees or keeps them.
 *  - Calls are asynchronous and ordered on `stream` (NULL = the legacy default stream).
 *    Arguments are validated on the host before anything is launched. A non-HSA_OK return
 *    means nothing was launched, except for HSA_ERR_CUDA, which reports a failed launch.
 *  - Conditions the host cannot check (an index past the visible length, a write past the
 *    capacity, a wait that timed out) are skipped on the device and recorded as a flag in a
 *    per-device status word, which hsa_get_device_status() reads. No kernel traps.
 *  - Entry indices are int32 positions inside a request, counted from 0. -1 means "none".
 *  - Selected index sets are unordered as a contract; the kernels emit them ascending.
 *  - One workspace may not be used by two calls that overlap on the device. The workspace
 *    must be zero-filled before its first use (hsa_workspace_init does that); every call
 *    leaves it zero-filled again when it completes.
 *
 * Cache layout (one buffer set per KV-source layer; SoA, request-major, `cap` = capacity):
 *   kv_q [batch][cap][256] u8   main-KV codes: 512 x E2M1. Byte j holds element 2j in its
 *                               low nibble and 2j+1 in its high nibble.
 *   kv_s [batch][cap][32]  u8   main-KV scales: one per 16 elements, E8M0 (2^(b-127)) or E4M3
 *                               ([890B] §三 事实一: 288 B per entry).
 *   ik_q [batch][cap][64]  u8   indexer-K codes: 128 x E2M1 in "fragment order". Stored byte
 *                               16t + 2s + i (t, i in {0..3}x{0,1}, s in 0..7) holds logical
 *                               byte 8s + 2t + i, i.e. elements 16s + 4t + 2i (low nibble) and
 *                               16s + 4t + 2i + 1 (high nibble).
 *   ik_s [batch][cap][4]   u8   indexer-K scales: E8M0, one per 32 elements
 *                               ([890B] §三 事实二: 68 B per entry).
 *   356 B per entry in total; 890 B/token over the 3 ratio-2 sources and the ratio-1 source.
 * The pages fix the value formats, not the byte order. The fragment order of ik_q lets the
 * scoring kernel read each thread's operands with one 16-byte load and keep every tensor-core
 * k-step inside one 32-element scale group.
 */
#ifndef HSA_H
#define HSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define HSA_API __attribute__((visibility("default")))
#else
#define HSA_API
#endif

#define HSA_ABI_VERSION 3

#define HSA_D_LATENT 512      /* main-KV latent width (head_dim)          [890B] §三 */
#define HSA_D_INDEX 128       /* indexer head dim (index_head_dim)        [890B] §三 */
#define HSA_H_INDEX 16        /* indexer heads                                      */
#define HSA_H_ATTN 64         /* attention query heads                    [ARCH] §1  */
#define HSA_TOPK 512          /* index_topk                               [890B] 注意力实际有多稀 */
#define HSA_CAND_BLOCKS 2048  /* candidate_topk_blocks                    [890B] §二 */
#define HSA_BLOCK 8           /* candidate_block_size                     [890B] §二 */
#define HSA_POOL_SLOTS 16384  /* 2048 x 8 candidate positions             [CED] Figure 5 */
#define HSA_POOL_TAIL_SLOTS 160 /* extra pool slots with HSA_CACHE_POOL_TAIL (<= 17 window blocks) */
#define HSA_SWA_W 128         /* sliding_window                           [890B] §二 */
#define HSA_MAX_NQ 8          /* query tokens per request per call (draft block 5 fits) */
#define HSA_MAX_VIS (1 << 20) /* longest visible context per query (1M, [ARCH] §1 table) */
#define HSA_ROPE_DIMS 64      /* rotary dims of the latent: its last 64 ([ARCH] §7: 448 NoPE + 128 B RoPE) */
#define HSA_ROPE_THETA 160000.0 /* RoPE base of the compressed latent       [ARCH] §3.2 */

typedef struct CUstream_st* hsa_stream_t; /* identical to cudaStream_t */

typedef enum {
  HSA_OK = 0,
  HSA_ERR_INVALID_ARG = 1, /* NULL pointer, bad enum or non-positive size           */
  HSA_ERR_SHAPE = 2,       /* sizes out of range (nq, capacity, max_vis, n_tokens)   */
  HSA_ERR_ALIGN = 3,       /* a pointer is not 16-byte aligned                       */
  HSA_ERR_WORKSPACE = 4,   /* workspace NULL or smaller than hsa_workspace_bytes()   */
  HSA_ERR_CUDA = 5,        /* a CUDA runtime call or kernel launch failed            */
  HSA_ERR_TIMEOUT = 6,     /* reported by hsa_get_device_status: a bounded wait ran out */
  HSA_ERR_UNSUPPORTED = 7  /* no sm_100-family device, or an unsupported option      */
} hsa_status;

typedef enum { HSA_SCALE_E8M0 = 0, HSA_SCALE_E4M3 = 1 } hsa_scale_fmt;

/* CSA2 layer modes ([CED] Figure 4; [ARCH] §3.2 table) */
typedef enum { HSA_MODE_FULL = 0, HSA_MODE_REINDEX = 1, HSA_MODE_REUSE = 2 } hsa_layer_mode;

/* Device status flags (bit mask returned by hsa_get_device_status) */
#define HSA_FLAG_INDEX_RANGE 1u   /* a top-k / pool index >= visible length or capacity was skipped */
#define HSA_FLAG_WRITE_RANGE 2u   /* a cache write past capacity was skipped                         */
#define HSA_FLAG_TIMEOUT 4u       /* a bounded device wait gave up                                  */

/* Cache flags (hsa_cache.flags) */
#define HSA_CACHE_ROPE 1u         /* the writer applies RoPE to the main-KV latent (see hsa_cache_write_compress) */
#define HSA_CACHE_POOL_TAIL 2u    /* index pools of this cache carry the window tail (see hsa_index_full) */

/* Caller-owned cache descriptor. All four buffers are device memory, 16-byte aligned. */
typedef struct {
  int32_t batch;        /* requests                                     */
  int32_t ratio;        /* compression ratio m of the writer: 1 or 2    */
  int64_t capacity;     /* entries per request; a multiple of 8         */
  int32_t kv_scale_fmt; /* hsa_scale_fmt of kv_s                        */
  int32_t flags;        /* HSA_CACHE_* bits; unknown bits are rejected  */
  uint8_t* kv_q;
  uint8_t* kv_s;
  uint8_t* ik_q;
  uint8_t* ik_s;
} hsa_cache;

/* Per-step arguments of hsa_schedule_step. Arrays indexed by layer slot l in [0, n_layers)
 * are HOST arrays of DEVICE pointers. */
typedef struct {
  int32_t n_layers;             /* e.g. 20 for decoder layers 20..39                       */
  int32_t nq;                   /* query tokens per request                                */
  const int32_t* modes;         /* host [n_layers] hsa_layer_mode; slot 0 must be FULL     */
  const void* const* q_idx;     /* [n_layers] -> bf16 [B][nq][16][128]; NULL for Reuse     */
  const float* const* w_idx;    /* [n_layers] -> f32 [B][nq][16]; NULL for Reuse           */
  const void* const* q_attn;    /* [n_layers] -> bf16 [B][nq][64][512]                     */
  const uint8_t* const* swa;    /* [n_layers] -> e4m3 [B][W+nq-1][512]                     */
  float* const* out;            /* [n_layers] -> f32 [B][nq][64][512]                      */
  int32_t* const* topk;         /* [n_layers] -> i32 [B][nq][512] for Full/Reindex slots;
                                   ignored for Reuse slots, which read the latest producer  */
  int32_t* pool;                /* i32 [B][nq][16384] (16544 with HSA_CACHE_POOL_TAIL), written by the Full slot */
  const int32_t* vis;           /* i32 [B][nq] visible lengths                              */
  int64_t max_vis;              /* host upper bound of vis                                  */
  float sm_scale;               /* softmax scale applied to q.k                             */
} hsa_step_args;

/* Library ABI version (HSA_ABI_VERSION). Host only. */
HSA_API int32_t hsa_abi_version(void);

/* Human-readable name of a status code. Host only; never NULL. */
HSA_API const char* hsa_status_string(hsa_status s);

/* Workspace bytes that hsa_index_full / hsa_index_reindex / hsa_sparse_attn_decode /
 * hsa_schedule_step need for `batch` requests of `nq` queries and visible lengths up to
 * `max_vis`. Host only; returns 0 for invalid sizes. */
HSA_API size_t hsa_workspace_bytes(int32_t batch, int32_t nq, int64_t max_vis);

/* Zero-fill a workspace (a cudaMemsetAsync on `stream`). */
HSA_API hsa_status hsa_workspace_init(void* ws, size_t ws_bytes, hsa_stream_t stream);

/* Compressed-cache write ([890B] §四.1 and §三; [ARCH] §3.2 "Z（压缩权重）的计算" and §7;
 * [CED] CSA2: the compressor keeps no overlap window and no absolute position encoding, and
 * indexer K is projected from the main-KV entry).
 * For each request b, token group i (m = cache->ratio consecutive tokens) becomes entry
 * start_entry[b] + i:
 *   m = 2: per channel c, p = softmax(wgate[2i][c], wgate[2i+1][c]), latent = p0 x0 + p1 x1 (fp32);
 *   m = 1: latent = wkv[i] (there is no gating path);
 *   latent <- RMSNorm(latent) (eps 1e-6, unit gain); K = latent . w_idx (512x128, fp32
 *   accumulate) <- FP4 group-32 E8M0; main KV <- FP4 group-16 with the cache's scale format, of
 *   the latent itself or, with HSA_CACHE_ROPE, of the latent with its last 64 dims rotated
 *   ([ARCH] §3.2: RMSNorm, then the no-RoPE version, then compressed RoPE with theta = 160000,
 *   then FP4; the indexer K is projected from the no-RoPE version): pair (448 + 2k, 449 + 2k),
 *   k = 0..31, turns by the entry's position (start_entry[b] + i) times theta^(-k/32) radians,
 *   (a, b) -> (a cos - b sin, a sin + b cos).
 * Scale rule: the smallest scale s (a power of two for E8M0, an E4M3 value otherwise) with
 * 6 s >= group amax. Codes are E2M1, round to nearest even, and -0 is stored as +0.
 *   wkv        bf16 [B][n_tokens][512]
 *   wgate      bf16 [B][n_tokens][512]; NULL iff ratio == 1
 *   w_idx      bf16 [512][128]
 *   n_tokens   tokens per request (a trailing group with fewer than m tokens is not written)
 *   start_entry  i64 [B] device; NULL means 0 for every request
 * Entries that would land at or past `capacity` are skipped and flagged HSA_FLAG_WRITE_RANGE. */
HSA_API hsa_status hsa_cache_write_compress(const hsa_cache* cache, const void* wkv, const void* wgate,
                                    const void* w_idx, int64_t n_tokens, const int64_t* start_entry,
                                    hsa_stream_t stream);

/* Full-mode indexer ([CED] Figure 5 left/middle; [ARCH] §3.3 建池 and 时序澄清; [10100]).
 * For each request b and query i (visible length vis[b][i] <= max_vis <= capacity):
 *   s_t = sum_h w[b][i][h] * ReLU(q[b][i][h] . k_t) over t < vis, with k_t the dequantised
 *   indexer K. From this one pass, two selections side by side:
 *   topk_out[b][i][0..512): the positions of the min(512, vis) largest s_t, ascending, -1 padded;
 *   pool_out[b][i][0..16384): the min(2048, ceil(vis/8)) blocks of 8 (aligned to position 0)
 *   with the largest block max, in ascending block order. Each block contributes 8 slots
 *   8b..8b+7, positions >= vis are -1, and unused slots are -1.
 * Ties go to the lower position or block. Scores are fp32 (tensor-core f16 products, fp32 sums).
 * With HSA_CACHE_POOL_TAIL in cache->flags ([ARCH] §3.3 旁路与边界: the newest tokens of the
 * sliding window skip the funnel and join the expanded pool at its tail), pool rows have
 * HSA_POOL_SLOTS + HSA_POOL_TAIL_SLOTS slots: the blocks holding positions [vis - 128, vis) join
 * the selected blocks, still as ascending 8-slot runs, and a window block the selection did not
 * pick keeps only its positions >= vis - 128 (its other slots are -1).
 *   q      bf16 [B][nq][16][128]      w   f32 [B][nq][16]      vis  i32 [B][nq]
 *   ws     workspace of at least hsa_workspace_bytes(B, nq, max_vis) bytes */
HSA_API hsa_status hsa_index_full(const hsa_cache* cache, const void* q, const float* w, const int32_t* vis,
                          int32_t nq, int64_t max_vis, int32_t* topk_out, int32_t* pool_out,
                          void* ws, size_t ws_bytes, hsa_stream_t stream);

/* Reindex-mode indexer ([CED] Figure 5 right; [ARCH] §3.3 池内过滤; [COST] §3.2).
 * Scores only the pool slots (pool[b][i][j] in [0, vis), others skipped) with this layer's
 * q and w, and writes the positions of the min(512, #valid) best, ascending, -1 padded.
 *   pool   i32 [B][nq][16384] as written by hsa_index_full ([B][nq][16544] with HSA_CACHE_POOL_TAIL)
 *   ws     workspace of at least hsa_workspace_bytes(B, nq, max_vis) bytes, checked like the
 *          other calls' so that one workspace serves every call; this call does not touch it
 *          (its CTAs exchange their candidates through distributed shared memory) */
HSA_API hsa_status hsa_index_reindex(const hsa_cache* cache, const void* q, const float* w, const int32_t* vis,
                             int32_t nq, int64_t max_vis, const int32_t* pool, int32_t* topk_out,
                             void* ws, size_t ws_bytes, hsa_stream_t stream);

/* Size of the fixed device array behind hsa_index_full_noalloc: 64 MiB on every device that
 * loads the library, held until the process exits. */
#define HSA_NOALLOC_SCRATCH_BYTES (64ull << 20)

/* The Full-mode indexer without a caller workspace. The pages have no counterpart for this
 * entry point; it is a convenience of this library for callers that cannot allocate device
 * memory: a plugin that may only touch the buffers it is handed, code running inside a memory
 * arena an inference server planned in advance, or a latency-critical loop that must never wait
 * on an allocator. Arguments, outputs and results are those of hsa_index_full without ws and
 * ws_bytes. The scratch the two Full kernels need lives in a fixed array of
 * HSA_NOALLOC_SCRATCH_BYTES inside the library. Limits and behaviour:
 *  - sizes whose Full scratch exceeds the array (about 41 B per row and visible position, e.g.
 *    batch 32 x 1 query x 131,072 positions fits) return HSA_ERR_WORKSPACE; nothing is launched;
 *  - the first call on a device looks up the array's address on that device; make that first
 *    call before any stream capture;
 *  - every call shares the array: each one clears the part that must start at zero with a
 *    cudaMemsetAsync on `stream` before its kernels, and two calls that overlap on the GPU (other
 *    streams, other threads) race on it;
 *  - it calls no cudaMalloc / cudaFree and no allocating library routine.
 * Other errors are those of hsa_index_full. */
HSA_API hsa_status hsa_index_full_noalloc(const hsa_cache* cache, const void* q, const float* w, const int32_t* vis,
                                          int32_t nq, int64_t max_vis, int32_t* topk_out, int32_t* pool_out,
                                          hsa_stream_t stream);

/* Sparse attention ([CED] Figure 4: Selected Main KV ⊕ SWA KV -> Core Attention;
 * [890B] 注意力实际有多稀: 512 + 128 = 640 positions; [ARCH] §7: dequantise before attention).
 * For request b, query i and head h:
 *   o = sum_j softmax_j(sm_scale * q_h . k_j) k_j, over the keys j = the main-KV entries
 *   topk[b][i][*] in [0, vis) and then SWA rows r in [i, i+128) of swa[b] whose position
 *   vis - 128 + (r - i) is >= 0. K = V = the 512-d latent. With no keys the output is 0.
 *   q     bf16 [B][nq][64][512]     topk  i32 [B][nq][512]     swa  e4m3 [B][128+nq-1][512]
 *   out   f32  [B][nq][64][512]
 *   ws    workspace of at least hsa_workspace_bytes(B, nq, max_vis) bytes, 16-byte aligned; it
 *         carries the partial outputs of the 4 key slices of each (b, i) between the CTAs that
 *         combine them, and needs no initialisation */
HSA_API hsa_status hsa_sparse_attn_decode(const hsa_cache* cache, const void* q, const int32_t* topk,
                                  const uint8_t* swa, const int32_t* vis, int32_t nq, int64_t max_vis,
                                  float sm_scale, float* out, void* ws, size_t ws_bytes,
                                  hsa_stream_t stream);

/* One decode step over consecutive layer slots ([ARCH] §3.3: 1 full score + 4 pool rescores +
 * 15 inherits; [COST] §3.1; [CED] Figure 4). Slot l runs its indexer if FULL (which also
 * writes the pool) or REINDEX, then attention with the latest indices. Every layer owns its
 * cache: `caches` is a HOST array of n_layers descriptors, and slot l scores caches[l]'s
 * indexer K (Full, Reindex) and attends over caches[l]'s main KV. Indices are positions, so an
 * inherited top-k or the Full slot's pool addresses the same tokens in every layer's cache.
 * The caches share batch and ratio and each holds at least max_vis entries (HSA_ERR_SHAPE
 * otherwise); a slot may repeat another's descriptor. Everything is stream-ordered, with no
 * host synchronisation. The step's inputs (q_attn, swa, q_idx, w_idx,
 * vis, pool when the first slot is not FULL) must be complete before the call's work starts on
 * `stream` and must not alias anything the step writes (out, topk, pool, ws): the attention
 * kernels fetch their queries and SWA rows, and the Reindex kernels their queries, weights and
 * pool rows, while the previous kernel of the step drains. */
HSA_API hsa_status hsa_schedule_step(const hsa_cache* caches, const hsa_step_args* args, void* ws,
                             size_t ws_bytes, hsa_stream_t stream);

/* Limit of the kernels' bounded waits (for a copy or a tensor-core result that does not arrive),
 * in nanoseconds, for launches made after the call from any thread, on every device. A wait that
 * runs out sets HSA_FLAG_TIMEOUT; the kernel then skips the work that needed it, waits (again
 * bounded) for its own copies and tensor-core work in flight, frees its tensor memory and
 * finishes, so the context stays usable. 0 restores the default, 2 s. Host only; no error. */
HSA_API hsa_status hsa_set_wait_limit(uint64_t ns);

/* Test hook for failure detection. The next hsa_index_full call (on any device or thread)
 * withholds one indexer-K copy of its scan kernel: the first CTA's last pipeline stage is never
 * filled, so that stage's consumer warps wait until the limit of hsa_set_wait_limit runs out,
 * set HSA_FLAG_TIMEOUT, skip the stage and finish with no copy or tensor-core work in flight.
 * That call's outputs are invalid; the workspace and every later call are unaffected. Host only. */
HSA_API hsa_status hsa_debug_stall_next_scan(void);

/* Synchronise `stream`, return the device status flags (HSA_FLAG_*) in *flags and clear them.
 * Returns HSA_ERR_TIMEOUT if HSA_FLAG_TIMEOUT is set, else HSA_OK or HSA_ERR_CUDA. */
HSA_API hsa_status hsa_get_device_status(hsa_stream_t stream, uint32_t* flags);

#ifdef __cplusplus
}
#endif
#endif /* HSA_H */
