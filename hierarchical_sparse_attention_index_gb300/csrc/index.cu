// Full-mode indexer kernels: FP4 indexer-K scoring over every visible position and the exact
// top-k selections behind it ([CED] Figure 5; [ARCH] §3.3; [COST] §3.2; [10100] 层次化稀疏索引器).
// The Reindex pass has its own fused kernel (reindex.cu).
//
// Scoring, s_t = sum_h w_h ReLU(q_h . k_t):
//  - One producer warp streams 512-entry stages of indexer K into a 3-deep shared-memory ring
//    with bulk async copies. Sixteen consumer warps score them.
//  - Each consumer thread reads its 16-byte chunk of an entry with one shared load. That chunk
//    holds the entry's bytes in "fragment order" (include/hsa.h). The thread converts E2M1 pairs
//    to f16x2 with the hardware cvt and feeds them straight into m16n8k16 tensor-core MMAs as
//    the A operand (rows = entries, k = dims, n = heads).
//  - Every k-step lies inside one 32-dim scale group, so the E8M0 scale is applied exactly in
//    fp32 to the per-group accumulator. The query is converted once per segment to f16, after a
//    per-head power-of-two shift that keeps its largest element in [2^14, 2^15). The shift is
//    folded back into the head weight.
//  - The epilogue fuses the ReLU-weighted head sum, the visibility mask and the 8-entry block
//    max ([ARCH] §3.3 块 max 是上界). It stores each score and each block max, and counts the
//    block maxima in a 4096-bin histogram of the top 12 bits of their order keys (one count per
//    block; positions are not histogrammed).
// Selection (exact; ties to the lower index), one CTA per (request, query) row, from the block
// maxima alone plus 4,096 scores ([ARCH] §3.3 时序澄清: both top-k's come from the one score
// pass):
//  - the histogram gives the threshold bins of the block top-2048 (the pool) and of the block
//    top-512; one pass over the row's block maxima takes the blocks above each threshold bin
//    and lists those inside it, and an exact cut among the listed ones completes both sets;
//  - the position top-512 lies inside the positions of the top-512 blocks: a block ranked
//    below them has at least 512 positions ranked above all of its own (each better block's
//    maximum), so none of its positions can be in the top 512. The kernel reads the 4,096
//    scores of those blocks and cuts the exact top-512 among them;
//  - the pool (blocks expanded to 8 slots) and the top-512 are written in ascending order, and
//    the row's histogram is cleared for the next call.
#include <algorithm>

#include "hsa_common.cuh"
#include "hsa_hist.cuh"
#include "hsa_internal.h"
#include "hsa_score.cuh"

namespace hsa {
namespace {

constexpr int kChunk = kScanChunk;
constexpr int kMaxStages = 4;
constexpr int kConsumerWarps = 16;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kScanThreads = kConsumers + 32;
constexpr int kCodesBytes = kChunk * 64;
constexpr int kScaleBytes = kChunk * 4;
constexpr int kFlushItems = 960;   // packed 16-bit histogram counters (64 blocks per item): flush before 65536

struct ScanSmemLayout {
  int nst, nlr;
  size_t codes, scales, bfrag, wsc, hist, sfl, bars, misc, total;
};

__host__ __device__ inline ScanSmemLayout scan_smem_layout(int nq) {
  ScanSmemLayout L;
  const int nql = nq;
  L.nst = (nql <= 2) ? 3 : (nql <= 5 ? 2 : 1);
  L.nlr = nq;                          // one block-max histogram per query
  size_t o = 0;
  L.codes = o;   o += (size_t)L.nst * kCodesBytes;
  L.scales = o;  o += (size_t)L.nst * kScaleBytes;
  L.bfrag = o;   o += (size_t)nql * 2 * 8 * 32 * 2 * 4;
  L.wsc = o;     o += (size_t)nql * 16 * 4;
  L.hist = o;    o += (size_t)L.nlr * (kHistBins / 2) * 4;
  L.sfl = o;     o += (size_t)kConsumerWarps * 32 * 16;   // per warp: its 32 rows' 4 group scales as floats
  L.bars = o;    o += 2 * kMaxStages * 8;
  L.misc = o;    o += 256;
  L.total = o;
  return L;
}

// A segment is one request (its nq queries share the request's indexer K); kOneQuery: nq == 1.
template <bool kOneQuery>
__global__ void __maxnreg__(96) index_scan_kernel(const ScanParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const ScanSmemLayout L = scan_smem_layout(p.nq);
  const int nql = kOneQuery ? 1 : p.nq;
  const int nst = kOneQuery ? 3 : L.nst;   // compile-time where it can be (scan_smem_layout)
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
  int* misc = reinterpret_cast<int*>(smem + L.misc);   // [0] abort, [2..9] vis
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + kMaxStages);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // contiguous item range of this CTA
  const int64_t per = ((int64_t)p.total_items + gridDim.x - 1) / gridDim.x;
  const int i0 = (int)imin64((int64_t)blockIdx.x * per, p.total_items);
  const int i1 = (int)imin64((int64_t)i0 + per, p.total_items);

  if (tid == 0) {
    for (int s = 0; s < nst; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, kConsumerWarps);
    }
    misc[0] = 0;
    fence_mbar_init();
  }
  {
    uint32_t* h = reinterpret_cast<uint32_t*>(smem + L.hist);
    for (int i = tid; i < L.nlr * (kHistBins / 2); i += kScanThreads) h[i] = 0;
  }
  __syncthreads();
  griddep_wait();
  griddep_launch_dependents();
  if (i0 >= i1) return;

  const int cps = p.chunks_per_seg;

  if (warp == kConsumerWarps) {
    // ---------------------------------------------------------------- producer warp
    // filled[s] / fph[s]: whether stage s was ever filled and the parity of its last fill. A wait
    // that gives up flags the status, stops the stream and falls through to the drain: the CTA
    // never exits with one of its copies still in flight.
    bool filled[kMaxStages] = {false, false, false, false};
    uint32_t fph[kMaxStages] = {0u, 0u, 0u, 0u};
    int s = 0, round = 0, seg = i0 / cps, c = i0 % cps;
    for (int it = i0; it < i1; ++it) {
      if (round > 0) {
        if (!mbar_wait(empty0 + 8 * s, (round - 1) & 1, p.wait_ns)) {
          flag_status(p.status, HSA_FLAG_TIMEOUT);
          *reinterpret_cast<volatile int*>(misc) = 1;
          break;
        }
      }
      const uint32_t full = full0 + 8 * s;
      const uint32_t dcodes = smem_u32(smem + L.codes + (size_t)s * kCodesBytes);
      const uint32_t dscales = smem_u32(smem + L.scales + (size_t)s * kScaleBytes);
      // test hook (hsa_debug_stall_next_scan): CTA 0 withholds its last stage, whose consumers
      // then wait in vain until the limit runs out
      const bool withhold = p.stall_last && blockIdx.x == 0 && it == i1 - 1;
      {
        int vmax = 0;
        for (int q = 0; q < p.nq; ++q) vmax = max(vmax, __ldg(p.vis + seg * p.nq + q));
        vmax = (int)imin64(vmax, p.cap);
        const int p0 = c * kChunk;
        const int n = max(0, min(kChunk, vmax - p0));
        if (lane == 0 && !withhold) {
          if (n > 0) {
            const int nc = (int)imin64((n + 7) & ~7, p.cap - p0);
            mbar_arrive_expect_tx(full, (uint32_t)nc * 68u);
            const int64_t e0 = (int64_t)seg * p.cap + p0;
            // indexer K is read once per Full call: evict it first, so that the scores the
            // selection reads next stay in L2
            const uint64_t pol = l2_policy_evict_first();
            bulk_g2s_hint(dcodes, p.ik_q + e0 * 64, (uint32_t)nc * 64u, full, pol);
            bulk_g2s_hint(dscales, p.ik_s + e0 * 4, (uint32_t)nc * 4u, full, pol);
          } else {
            mbar_arrive(full);
          }
        }
        if (!withhold) {
          filled[s] = true;
          fph[s] = (uint32_t)round & 1u;
        }
      }
      if (++s == nst) {
        s = 0;
        ++round;
      }
      if (++c == cps) {
        c = 0;
        ++seg;
      }
    }
    // drain: every copy this warp issued has landed (immediate unless a consumer gave up early)
    for (int st = 0; st < nst; ++st)
      if (filled[st] && !mbar_wait(full0 + 8 * st, fph[st], p.wait_ns)) flag_status(p.status, HSA_FLAG_TIMEOUT);
    return;
  }

  // ------------------------------------------------------------------ consumer warps
  const int g = lane >> 2, t = lane & 3;
  uint32_t* hist_sm = reinterpret_cast<uint32_t*>(smem + L.hist);
  uint32_t* bfrag = reinterpret_cast<uint32_t*>(smem + L.bfrag);
  float* wsc = reinterpret_cast<float*>(smem + L.wsc);
  int* svis = misc + 2;

  uint32_t B[2][8][2];   // query fragments of the current query (registers)
  float wr[2][2];
  int cur_seg = -1, since_flush = 0;

  auto flush_hist = [&](int seg) {
    named_bar_sync(1, kConsumers);
    for (int lr = 0; lr < L.nlr; ++lr) {
      uint32_t* gh = p.hist + (size_t)(seg * p.nq + lr) * kHistBins;
      uint32_t* sh = hist_sm + lr * (kHistBins / 2);
      for (int i = tid; i < kHistBins / 2; i += kConsumers) {
        const uint32_t v = sh[i];
        if (v) {
          if (v & 0xFFFFu) atomicAdd(gh + 2 * i, v & 0xFFFFu);
          if (v >> 16) atomicAdd(gh + 2 * i + 1, v >> 16);
          sh[i] = 0;
        }
      }
    }
    named_bar_sync(1, kConsumers);
  };

  auto load_segment = [&](int seg) {
    named_bar_sync(1, kConsumers);
    for (int ql = 0; ql < nql && tid < 256; ++ql) {
      const int row = seg * p.nq + ql;
      stage_query(p.q + (size_t)row * kHIdx * kDIdx, p.w + (size_t)row * kHIdx, bfrag + ql * kQFragWords,
                  wsc + ql * kQWeights, tid);
      if (tid < 8 && tid == ql) svis[ql] = (int)imin64(__ldg(p.vis + row), p.cap);
    }
    named_bar_sync(1, kConsumers);
  };

  auto load_query_regs = [&](int ql) { load_query_frags(bfrag + ql * kQFragWords, wsc + ql * kQWeights, lane, B, wr); };

  // Stage index, ring parity and (segment, chunk) advance incrementally. Segment changes and
  // histogram flushes are the same for every consumer warp, so the named barriers inside them
  // stay matched; a wait that times out flags the status and that warp skips its remaining
  // stages (no early exit, so the barriers still match).
  int s = 0, seg = i0 / cps, c = i0 % cps;
  uint32_t ph = 0;
  bool dead = false;
  int vmax_seg = 0;                // Full: visible rows of the current request (max over its queries)

  for (int it = i0; it < i1; ++it) {
    if (seg != cur_seg) {
      if (cur_seg >= 0) flush_hist(cur_seg);
      cur_seg = seg;
      since_flush = 0;
      load_segment(seg);
      if (nql == 1) load_query_regs(0);
      int vmax = 0;
      for (int q = 0; q < nql; ++q) vmax = max(vmax, svis[q]);
      vmax_seg = vmax;             // svis is already capped at the capacity
    } else if (since_flush >= kFlushItems) {
      flush_hist(seg);
      since_flush = 0;
    }
    ++since_flush;
    if (!dead && *reinterpret_cast<volatile int*>(misc) != 0) dead = true;
    if (!dead && !mbar_wait(full0 + 8 * s, ph, p.wait_ns)) {
      flag_status(p.status, HSA_FLAG_TIMEOUT);
      *reinterpret_cast<volatile int*>(misc) = 1;
      dead = true;
    }
    const uint32_t codes = smem_u32(smem + L.codes) + (uint32_t)s * kCodesBytes;
    const uint32_t scales = smem_u32(smem + L.scales) + (uint32_t)s * kScaleBytes;
    const int row_off = warp * 32;   // first row of this warp inside the stage
    const int nrows = dead ? 0 : max(0, min(kChunk, vmax_seg - c * kChunk));

    if (warp * 32 < nrows) {
      const uint32_t sf_base = smem_u32(smem + L.sfl) + (uint32_t)warp * 512u;
      stage_group_scales(scales, row_off, sf_base, lane);
      // this lane's row after the reduce-scatter: rows 8t .. 8t+7 of the warp's 32 are the
      // 8-entry block t, one row per lane g
      const int r_mine = warp * 32 + 8 * t + g;
      for (int ql = 0; ql < nql; ++ql) {
        if (nql > 1) load_query_regs(ql);
        // both 16-row tiles are always scored, so the compiler can interleave their independent
        // convert and MMA chains (a conditional second tile serialised them: Full call 92.2 ->
        // 89.4 us); rows past the stage's data hold stale bytes and are masked just below
        float v = score_rows32(codes, row_off, sf_base, B, wr, lane);
        const bool ok = c * kChunk + r_mine < svis[ql];
        v = ok ? v : -INFINITY;
        {
          const int row = cur_seg * p.nq + ql;
          p.scores[(size_t)row * p.ld_s + c * kChunk + r_mine] = v;
          // 8-entry block max: block t of the warp is held by lanes g = 0..7 of column t
          float bm = v;
          bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 4));
          bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 8));
          bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 16));
          const int jb = ((c * kChunk + warp * 32) >> 3) + t;
          if (g == 0 && jb * 8 < svis[ql]) {
            p.blkmax[(size_t)row * p.ld_b + jb] = bm;
            const uint32_t bb = order_key(bm) >> kHistShift;
            atomicAdd(hist_sm + ql * (kHistBins / 2) + (bb >> 1), (bb & 1) ? 0x10000u : 1u);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * s);
    if (++s == nst) {
      s = 0;
      ph ^= 1u;
    }
    if (++c == cps) {
      c = 0;
      ++seg;
    }
  }
  if (cur_seg >= 0) flush_hist(cur_seg);
}

// ------------------------------------------------------------------ select
constexpr int kSelThreads = 512;
constexpr int kSelStage = 4096;     // threshold-bin candidates ranked from shared memory; more from L2
constexpr int kSelRankMax = 512;    // elements ranked by counting up to this many
constexpr int kTopBlocks = kTopK;   // the position top-512 lies inside the top-512 blocks
constexpr int kPosCand = kTopBlocks * kBlk;   // 4096 position candidates

// the smallest float whose order key is `key` (inverse of order_key)
__device__ __forceinline__ float key_to_float(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}
// (order key, inverted index): larger = better, ties to the lower index
__device__ __forceinline__ uint64_t sel_comp(float v, uint32_t idx) {
  return ((uint64_t)order_key(v) << 32) | (uint64_t)(~idx);
}

struct SelShared {
  uint32_t hist[kHistBins];
  uint64_t rk[kSelRankMax];
  int scr[128];
  uint64_t cut;
  int ncand[1];
  int n_rk;
};

// Completes an exact top-`need` among the C candidates comp(0..C-1) (distinct 64-bit
// composites, larger = better) whose bits under `mask` all equal `prefix`; on return a candidate
// c is taken iff (c & mask) >= prefix. Levels: a 4096-bin histogram of composite bits 51..40,
// then counting when at most kSelRankMax remain tied, else a radix select over bits 39..0 in
// 11-bit digits. All kSelThreads threads call it.
template <typename CompFn>
__device__ void cut_candidates(CompFn comp, int C, int need, SelShared& S, uint64_t& prefix, uint64_t& mask,
                               int tid) {
  const int lane = tid & 31, warp = tid >> 5;
  if (need >= C) return;             // every candidate is taken
  for (int i = tid; i < kHistBins; i += kSelThreads) S.hist[i] = 0u;
  __syncthreads();
  for (int i = tid; i < C; i += kSelThreads) {
    const uint64_t c = comp(i);
    if ((c & mask) == prefix) atomicAdd(S.hist + ((c >> 40) & 0xFFFu), 1u);
  }
  __syncthreads();
  const int tied = smem_threshold<kSelThreads>(S.hist, need, S.scr, S.scr + 64, tid);
  if (tied <= need) {                // every tied candidate is taken
    __syncthreads();
    return;
  }
  const int thr2 = S.scr[64];
  int need_r = need - S.scr[65];
  prefix |= (uint64_t)thr2 << 40;
  mask |= 0xFFFull << 40;
  const int C2 = (int)S.hist[thr2];
  __syncthreads();                   // S.scr and S.hist read everywhere
  if (need_r >= C2) return;          // the whole bin is taken
  if (C2 <= kSelRankMax) {
    // few left: the need_r-th largest of them by counting
    if (tid == 0) S.n_rk = 0;
    __syncthreads();
    for (int i0 = warp * 32; i0 < C; i0 += kSelThreads) {
      const int i = i0 + lane;
      const uint64_t c = (i < C) ? comp(i) : 0ull;
      const bool in = (i < C) && (c & mask) == prefix;
      const int j = warp_append(in, &S.n_rk, lane);
      if (in) S.rk[j] = c;
    }
    __syncthreads();
    for (int i = tid; i < C2; i += kSelThreads) {
      const uint64_t ci = S.rk[i];
      int better = 0;
      for (int j = 0; j < C2; ++j) better += (S.rk[j] > ci) ? 1 : 0;
      if (better == need_r - 1) S.cut = ci;
    }
    __syncthreads();
    prefix = S.cut;
    mask = ~0ull;
    return;
  }
  // many tied in 24 key bits: radix select over composite bits 39..0
  const int shifts[4] = {29, 18, 7, 0};
  const int widths[4] = {11, 11, 11, 7};
  constexpr int kPerD = 2048 / kSelThreads;        // 4 digit bins per thread, high first
  for (int d = 0; d < 4; ++d) {
    const int sh = shifts[d];
    const uint32_t wm = (1u << widths[d]) - 1u;
    for (int i = tid; i < 2048; i += kSelThreads) S.hist[i] = 0u;
    __syncthreads();
    for (int i = tid; i < C; i += kSelThreads) {
      const uint64_t c = comp(i);
      if ((c & mask) == prefix) atomicAdd(S.hist + ((c >> sh) & wm), 1u);
    }
    __syncthreads();
    const int dtop = 2048 - kPerD * (tid + 1);
    int dc[kPerD], dl = 0;
#pragma unroll
    for (int k = 0; k < kPerD; ++k) {
      dc[k] = (int)S.hist[dtop + kPerD - 1 - k];
      dl += dc[k];
    }
    int dtot;
    const int dex = excl_scan(dl, S.scr, 1, kSelThreads, &dtot, tid);
    if (dex < need_r && dex + dl >= need_r) {
      int run = dex;
#pragma unroll
      for (int k = 0; k < kPerD; ++k) {
        if (run + dc[k] >= need_r) {
          S.scr[80] = dtop + kPerD - 1 - k;
          S.scr[81] = run;
          S.scr[82] = dc[k];
          break;
        }
        run += dc[k];
      }
    }
    __syncthreads();
    need_r -= S.scr[81];
    prefix |= (uint64_t)S.scr[80] << sh;
    mask |= (uint64_t)wm << sh;
    const bool all_in = (S.scr[82] == need_r);
    __syncthreads();
    if (all_in) break;
  }
}

// Ascending emission of a bitmap's set bits (bit i = element i): each thread owns the words
// [w0, w1); returns the output offset of its first set bit and the total in *total.
__device__ __forceinline__ int bitmap_offsets(const uint32_t* bitmap, int w0, int w1, int* scr, int tid,
                                              int* total) {
  int cnt = 0;
  for (int i = w0; i < w1; ++i) cnt += __popc(bitmap[i]);
  return excl_scan(cnt, scr, 1, kSelThreads, total, tid);
}

// One 2-CTA cluster per (request, query) row. CTA 0 selects the block top-2048 and writes the
// pool; CTA 1 selects the block top-512 and then the position top-512 among their positions.
// Both read the row's block-max histogram; CTA 1 clears it once CTA 0 has read it (the cluster
// barrier's arrive and wait are split around the work).
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kSelThreads) select_kernel(const SelectParams p) {
  extern __shared__ __align__(16) uint8_t fsm_raw[];
  const int tid = threadIdx.x;
  const int rank = (int)cluster_rank();
  const int row = blockIdx.x >> 1;
  __shared__ SelShared S;
  __shared__ int s_thr, s_above, s_total;
  __shared__ int s_tblk[kTopBlocks];
  __shared__ uint32_t s_psel[kPosCand / 32];
  griddep_wait();
  griddep_launch_dependents();
  const float* bm = p.blkmax + (size_t)row * p.ld_b;
  // The block pass's first batch of block maxima (eight float4 per thread) goes in flight with
  // the histogram loads instead of after the threshold is known. Its bound comes from max_vis
  // (the row stride ld_b covers it, rounded up to 64 blocks); chunks past this row's vis hold
  // values of no block and are masked by the block bound in the pass.
  constexpr int kIlp = 8;
  float4 v[kIlp];
  {
    const int nq4_max = (int)(((p.max_vis + kBlk - 1) / kBlk + 3) >> 2);
#pragma unroll
    for (int u = 0; u < kIlp; ++u) {
      const int c = u * kSelThreads + tid;
      v[u] = (c < nq4_max) ? __ldcg(reinterpret_cast<const float4*>(bm) + c) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  const int vis = (int)imin64(imax64(__ldg(p.vis + row), 0), p.max_vis);
  const int nb = (vis + kBlk - 1) / kBlk;
  const int nwb = (nb + 31) >> 5;                     // bitmap words
  const int K = rank ? kTopBlocks : kCandBlocks;
  uint32_t* bits = reinterpret_cast<uint32_t*>(fsm_raw);                 // [nwb4] selected blocks
  const int nwb4 = (nwb + 3) & ~3;
  uint64_t* cst = reinterpret_cast<uint64_t*>(bits + nwb4);             // [kSelStage] staged candidates
  int32_t* gcand = p.cand + (size_t)row * p.ld_cand + (size_t)rank * p.ld_b;   // candidates past the stage
  uint32_t* gh = p.hist + (size_t)row * kHistBins;

  // ---------------------------------------------------------------- 1. threshold bin of this CTA's block top-K
  {
    constexpr int kPer = kHistBins / kSelThreads;     // 8 bins per thread, high first
    const int top = kHistBins - kPer * (tid + 1);
    int cnt[kPer], local = 0;
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      cnt[k] = (int)__ldcg(gh + top + kPer - 1 - k);
      local += cnt[k];
    }
    int total;
    const int excl = excl_scan(local, S.scr, 1, kSelThreads, &total, tid);
    if (total <= K) {
      if (tid == 0) {
        s_thr = -1;
        s_above = total;
      }
    } else if (excl < K && excl + local >= K) {
      int run = excl;
#pragma unroll
      for (int k = 0; k < kPer; ++k) {
        if (run + cnt[k] >= K) {
          s_thr = top + kPer - 1 - k;
          s_above = run;
          break;
        }
        run += cnt[k];
      }
    }
    if (tid == 0) {
      s_total = total;
      S.ncand[0] = 0;
    }
    for (int i = tid; i < nwb4; i += kSelThreads) bits[i] = 0u;
  }
  cluster_arrive();                   // this CTA has read the histogram
  __syncthreads();
  if (rank == 0 && tid == 0 && s_total != nb) flag_status(p.status, HSA_FLAG_INDEX_RANGE);

  // ---------------------------------------------------------------- 2. one pass over the block maxima
  // Blocks above the threshold bin are taken at once; blocks in it are listed as candidates
  // (composites staged in shared memory, block indices in the workspace past the stage). Per
  // batch of 4,096 float4 (eight loads per thread; the next batch's loads are issued before this
  // one is classified), each thread counts its candidates and one block-wide exclusive scan
  // places them: no shared counter is contended.
  {
    const int thr = s_thr;
    // f_lo, the smallest float of the threshold bin: a block max below it is neither taken nor
    // listed, which one float compare decides for most blocks. The compare only filters: the
    // bin of a block that passes is decided on its order key (which tells -0 from +0). The
    // lowest keys of bins 0..7 are NaN patterns (-inf lies in bin 7): there the filter passes
    // everything, and NaN block maxima always pass, so the filter never changes a decision
    float f_lo = (thr < 0) ? -INFINITY : key_to_float((uint32_t)thr << kHistShift);
    if (f_lo != f_lo) f_lo = -INFINITY;
    const int nq4 = (nb + 3) >> 2;                    // float4 chunks
    int listed = 0;                                   // candidates of earlier batches (same in every thread)
    for (int c0 = 0; c0 < nq4; c0 += kIlp * kSelThreads) {
      float4 cur[kIlp];
#pragma unroll
      for (int u = 0; u < kIlp; ++u) cur[u] = v[u];
      if (c0 + kIlp * kSelThreads < nq4) {
#pragma unroll
        for (int u = 0; u < kIlp; ++u) {
          const int c = c0 + (kIlp + u) * kSelThreads + tid;
          v[u] = (c < nq4) ? __ldcg(reinterpret_cast<const float4*>(bm) + c) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      uint32_t candm[kIlp];
      int n = 0;
#pragma unroll
      for (int u = 0; u < kIlp; ++u) {
        const int c = c0 + u * kSelThreads + tid;
        const float f[4] = {cur[u].x, cur[u].y, cur[u].z, cur[u].w};
        uint32_t take = 0u;
        candm[u] = 0u;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          if (4 * c + k < nb && (f[k] >= f_lo || f[k] == 0.f || f[k] != f[k])) {
            const int bin = (int)(order_key(f[k]) >> kHistShift);
            if (thr < 0 || bin > thr) take |= 1u << k;
            else if (bin == thr) candm[u] |= 1u << k;
          }
        }
        if (take) atomicOr(bits + ((4 * c) >> 5), take << ((4 * c) & 31));
        n += __popc(candm[u]);
      }
      int total;
      int j = listed + excl_scan(n, S.scr, 1, kSelThreads, &total, tid);
      listed += total;
#pragma unroll
      for (int u = 0; u < kIlp; ++u) {
        const int c = c0 + u * kSelThreads + tid;
        const float f[4] = {cur[u].x, cur[u].y, cur[u].z, cur[u].w};
        uint32_t m = candm[u];
        while (m) {
          const int k = __ffs(m) - 1;
          m &= m - 1u;
          const int b = 4 * c + k;
          if (j < kSelStage) cst[j] = sel_comp(f[k], (uint32_t)b);
          else gcand[j - kSelStage] = b;
          ++j;
        }
      }
    }
    if (tid == 0) S.ncand[0] = listed;
  }
  __syncthreads();

  // ---------------------------------------------------------------- 3. cut the threshold bin, mark its taken blocks
  if (s_thr >= 0) {
    const int C = S.ncand[0];
    const int need = K - s_above;
    auto comp = [&](int i) -> uint64_t {
      if (i < kSelStage) return cst[i];
      const int b = __ldcg(gcand + (i - kSelStage));
      return sel_comp(__ldcg(bm + b), (uint32_t)b);
    };
    uint64_t prefix = (uint64_t)s_thr << 52, mask = 0xFFFull << 52;
    cut_candidates(comp, C, need, S, prefix, mask, tid);
    for (int i = tid; i < C; i += kSelThreads) {
      const uint64_t c = comp(i);
      if ((c & mask) >= prefix) {
        const uint32_t b = ~(uint32_t)c;
        atomicOr(bits + (b >> 5), 1u << (b & 31));
      }
    }
    __syncthreads();
  }

  const int per = (nwb + kSelThreads - 1) / kSelThreads;
  const int w0 = min(nwb, tid * per), w1 = min(nwb, w0 + per);
  if (rank == 0) {
    // ---------------------------------------------------------------- 4a. the pool, ascending
    // With the window tail ([ARCH] §3.3 旁路与边界) the blocks of positions [vis - W, vis) join
    // the selected ones; a window block the selection did not pick keeps only its window
    // positions. They are the row's last blocks, so ascending block order puts them at the tail.
    const int wlo = p.tail ? max(0, vis - kSwa) : vis;
    const int wb0 = p.tail ? wlo / kBlk : nb;         // first window block
    auto wmask = [&](int i) -> uint32_t {             // window blocks inside bitmap word i
      const int lo = max(wb0, 32 * i), hi = min(nb, 32 * i + 32);
      if (lo >= hi) return 0u;
      const uint32_t m = (hi - lo == 32) ? 0xFFFFFFFFu : ((1u << (hi - lo)) - 1u);
      return m << (lo - 32 * i);
    };
    int cnt = 0;
    for (int i = w0; i < w1; ++i) cnt += __popc(bits[i] | wmask(i));
    int totp;
    int o = excl_scan(cnt, S.scr, 1, kSelThreads, &totp, tid);
    const int max_runs = (int)(p.pool_ld / kBlk);
    int32_t* out = p.pool_out + (size_t)row * p.pool_ld;
    for (int i = w0; i < w1; ++i) {
      const uint32_t selw = bits[i];
      uint32_t m = selw | wmask(i);
      while (m) {
        const int bi = __ffs(m) - 1;
        m &= m - 1;
        const int blk = i * 32 + bi;
        const int lo = ((selw >> bi) & 1u) ? 0 : wlo;  // first position the run keeps
        if (o < max_runs) {
          const int q0 = blk * 8;
          int4 lo4, hi4;
          lo4.x = (q0 + 0 < vis && q0 + 0 >= lo) ? q0 + 0 : -1;
          lo4.y = (q0 + 1 < vis && q0 + 1 >= lo) ? q0 + 1 : -1;
          lo4.z = (q0 + 2 < vis && q0 + 2 >= lo) ? q0 + 2 : -1;
          lo4.w = (q0 + 3 < vis && q0 + 3 >= lo) ? q0 + 3 : -1;
          hi4.x = (q0 + 4 < vis && q0 + 4 >= lo) ? q0 + 4 : -1;
          hi4.y = (q0 + 5 < vis && q0 + 5 >= lo) ? q0 + 5 : -1;
          hi4.z = (q0 + 6 < vis && q0 + 6 >= lo) ? q0 + 6 : -1;
          hi4.w = (q0 + 7 < vis && q0 + 7 >= lo) ? q0 + 7 : -1;
          reinterpret_cast<int4*>(out + 8 * o)[0] = lo4;
          reinterpret_cast<int4*>(out + 8 * o)[1] = hi4;
        }
        ++o;
      }
    }
    for (int64_t j = 8 * (int64_t)min(totp, max_runs) + tid; j < p.pool_ld; j += kSelThreads) out[j] = -1;
    cluster_wait();
    return;
  }

  // ---------------------------------------------------------------- 4b. the top-512 blocks, ascending
  {
    int tott;
    int ot = bitmap_offsets(bits, w0, w1, S.scr, tid, &tott);
    for (int i = w0; i < w1; ++i) {
      uint32_t m = bits[i];
      while (m) {
        const int blk = i * 32 + __ffs(m) - 1;
        m &= m - 1;
        if (ot < kTopBlocks) s_tblk[ot] = blk;
        ++ot;
      }
    }
    if (tid == 0) S.ncand[0] = min(tott, kTopBlocks);
    for (int j = tid; j < kPosCand / 32; j += kSelThreads) s_psel[j] = 0u;
  }
  __syncthreads();

  // ---------------------------------------------------------------- 5. the position top-512 among those blocks
  // Candidate i is position 8 tblk[i / 8] + i % 8, so the list is in ascending position order.
  // Positions at or past vis get composite 0, below every score's.
  const int nt = S.ncand[0];
  const int U = nt * kBlk;
  uint64_t* pc = cst;                 // [4096] position composites (the stage is free now)
  {
    const float* sc = p.scores + (size_t)row * p.ld_s;
    if (tid < nt) {
      const int q0 = 8 * s_tblk[tid];
      const float4 a = __ldcg(reinterpret_cast<const float4*>(sc + q0));
      const float4 c = __ldcg(reinterpret_cast<const float4*>(sc + q0 + 4));
      const float f[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
#pragma unroll
      for (int j = 0; j < 8; ++j)
        pc[8 * tid + j] = (q0 + j < vis) ? sel_comp(f[j], (uint32_t)(q0 + j)) : 0ull;
    }
  }
  cluster_wait();                     // CTA 0 has read the histogram: clear it for the next call
#pragma unroll
  for (int k = 0; k < kHistBins / kSelThreads; ++k) gh[tid + k * kSelThreads] = 0u;
  __syncthreads();
  const int K2 = min(kTopK, vis);
  {
    auto comp = [&](int i) -> uint64_t { return pc[i]; };
    uint64_t prefix = 0ull, mask = 0ull;
    if (K2 < U) {
      // level 1 over the composites' top 12 bits, then cut_candidates inside the threshold bin
      for (int i = tid; i < kHistBins; i += kSelThreads) S.hist[i] = 0u;
      __syncthreads();
      for (int i = tid; i < U; i += kSelThreads) atomicAdd(S.hist + (int)(pc[i] >> 52), 1u);
      __syncthreads();
      smem_threshold<kSelThreads>(S.hist, K2, S.scr, S.scr + 64, tid);
      const int thr1 = S.scr[64], above1 = S.scr[65];
      __syncthreads();
      prefix = (uint64_t)thr1 << 52;
      mask = 0xFFFull << 52;
      cut_candidates(comp, U, K2 - above1, S, prefix, mask, tid);
    }
    for (int i = tid; i < U; i += kSelThreads)
      if (pc[i] != 0ull && (pc[i] & mask) >= prefix) atomicOr(s_psel + (i >> 5), 1u << (i & 31));
  }
  __syncthreads();
  {
    // 128 words of selection bits; thread tid < 128 owns word tid
    const int nw = (U + 31) >> 5;
    const int v0 = min(nw, tid), v1 = min(nw, tid + 1);
    int tot;
    int o = bitmap_offsets(s_psel, v0, v1, S.scr, tid, &tot);
    int32_t* out = p.topk_out + (size_t)row * kTopK;
    for (int i = v0; i < v1; ++i) {
      uint32_t m = s_psel[i];
      while (m) {
        const int k = i * 32 + __ffs(m) - 1;
        m &= m - 1;
        if (o < kTopK) out[o] = 8 * s_tblk[k >> 3] + (k & 7);
        ++o;
      }
    }
    for (int j = min(tot, kTopK) + tid; j < kTopK; j += kSelThreads) out[j] = -1;
  }
}
}  // namespace

template <bool kOneQuery>
cudaError_t launch_scan_variant(const ScanParams& p, int num_sms, cudaStream_t s) {
  const ScanSmemLayout L = scan_smem_layout(p.nq);
  auto kern = index_scan_kernel<kOneQuery>;
  cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(kern), L.total);
  if (e != cudaSuccess) return e;
  int per_sm = 1;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kScanThreads, L.total) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  int grid = num_sms * per_sm;
  if (grid > p.total_items) grid = p.total_items;
  if (grid < 1) grid = 1;
  return launch_pdl(kern, dim3(grid), dim3(kScanThreads), L.total, s, p);
}

cudaError_t launch_index_scan(const ScanParams& p, int num_sms, cudaStream_t s) {
  if (p.nq == 1) return launch_scan_variant<true>(p, num_sms, s);
  return launch_scan_variant<false>(p, num_sms, s);
}

cudaError_t launch_select(const SelectParams& p, cudaStream_t s) {
  const int rows = p.batch * p.nq;
  const int64_t nb = (std::max<int64_t>(p.max_vis, 1) + kBlk - 1) / kBlk;
  const int64_t nwb4 = ((nb + 31) / 32 + 3) & ~3;   // bitmap words
  const size_t smem = (size_t)nwb4 * 4 + (size_t)kSelStage * 8;
  cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(select_kernel), smem);
  if (e != cudaSuccess) return e;
  // one 2-CTA cluster per (request, query) row
  return launch_pdl(select_kernel, dim3((unsigned)(2 * rows)), dim3(kSelThreads), smem, s, p);
}

}  // namespace hsa
