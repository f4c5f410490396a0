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
//  - The epilogue fuses the ReLU-weighted head sum, the visibility mask, the 8-entry block max
//    ([ARCH] §3.3 块 max 是上界) and a 4096-bin histogram of the top 12 bits of each score's
//    order key. The last CTA to finish a request turns the histograms into the threshold bins
//    of the position top-512 and the block top-2048.
// Selection (exact; ties to the lower index), one 4-CTA cluster per (row, selection), each CTA
// streaming a quarter of the array: elements above the threshold bin are taken, elements in it
// become candidates, and after one cluster barrier a count or an 11-bit-digit radix select over
// (low key bits, inverted index) composites picks the remaining ones. Each quarter's bitmap is
// emitted in ascending order at its offset (blocks expanded into the candidate pool), and the
// workspace state is cleared.
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
constexpr int kFlushItems = 120;   // packed 16-bit histogram counters: flush before 65536 entries

struct ScanSmemLayout {
  int nst, nlr;
  size_t codes, scales, bfrag, wsc, hist, sfl, bars, misc, total;
};

__host__ __device__ inline ScanSmemLayout scan_smem_layout(int nq) {
  ScanSmemLayout L;
  const int nql = nq;
  L.nst = (nql <= 2) ? 3 : (nql <= 5 ? 2 : 1);
  L.nlr = 2 * nq;
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
  int* misc = reinterpret_cast<int*>(smem + L.misc);   // [0] abort, [1] last flag, [2..9] vis, [16..48) scratch
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
    int s = 0, round = 0, seg = i0 / cps, c = i0 % cps;
    for (int it = i0; it < i1; ++it) {
      if (round > 0) {
        if (!mbar_wait(empty0 + 8 * s, (round - 1) & 1)) {
          flag_status(p.status, HSA_FLAG_TIMEOUT);
          *reinterpret_cast<volatile int*>(misc) = 1;
          return;
        }
      }
      const uint32_t full = full0 + 8 * s;
      const uint32_t dcodes = smem_u32(smem + L.codes + (size_t)s * kCodesBytes);
      const uint32_t dscales = smem_u32(smem + L.scales + (size_t)s * kScaleBytes);
      {
        int vmax = 0;
        for (int q = 0; q < p.nq; ++q) vmax = max(vmax, __ldg(p.vis + seg * p.nq + q));
        vmax = (int)imin64(vmax, p.cap);
        const int p0 = c * kChunk;
        const int n = max(0, min(kChunk, vmax - p0));
        if (lane == 0) {
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
    return;
  }

  // ------------------------------------------------------------------ consumer warps
  const int g = lane >> 2, t = lane & 3;
  uint32_t* hist_sm = reinterpret_cast<uint32_t*>(smem + L.hist);
  uint32_t* bfrag = reinterpret_cast<uint32_t*>(smem + L.bfrag);
  float* wsc = reinterpret_cast<float*>(smem + L.wsc);
  int* svis = misc + 2;
  int* scratch = misc + 16;

  uint32_t B[2][8][2];   // query fragments of the current query (registers)
  float wr[2][2];
  int cur_seg = -1, seg_items = 0, since_flush = 0;

  auto flush_hist = [&](int seg) {
    named_bar_sync(1, kConsumers);
    for (int lr = 0; lr < L.nlr; ++lr) {
      const int grow = (seg * p.nq + (lr >> 1)) * 2 + (lr & 1);
      uint32_t* gh = p.hist + (size_t)grow * kHistBins;
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
    __threadfence();
    named_bar_sync(1, kConsumers);
  };

  auto finish_segment = [&](int seg, int nitems) {
    flush_hist(seg);
    if (tid == 0) {
      const unsigned old = atomicAdd(p.seg_done + seg, (unsigned)nitems);
      misc[1] = (old + (unsigned)nitems == (unsigned)cps) ? 1 : 0;
    }
    named_bar_sync(1, kConsumers);
    if (misc[1]) {
      __threadfence();
      for (int q = 0; q < p.nq; ++q) {
        const int row = seg * p.nq + q;
        compute_threshold<kConsumers>(p.hist + (size_t)(2 * row) * kHistBins, kTopK, p.state + 2 * row, scratch);
        compute_threshold<kConsumers>(p.hist + (size_t)(2 * row + 1) * kHistBins, kCandBlocks, p.state + 2 * row + 1,
                                      scratch);
      }
      if (tid == 0) p.seg_done[seg] = 0;
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
      if (cur_seg >= 0) finish_segment(cur_seg, seg_items);
      cur_seg = seg;
      seg_items = 0;
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
    ++seg_items;
    ++since_flush;
    if (!dead && *reinterpret_cast<volatile int*>(misc) != 0) dead = true;
    if (!dead && !mbar_wait(full0 + 8 * s, ph)) {
      flag_status(p.status, HSA_FLAG_TIMEOUT);
      *reinterpret_cast<volatile int*>(misc) = 1;
      dead = true;
    }
    const uint32_t codes = smem_u32(smem + L.codes) + (uint32_t)s * kCodesBytes;
    const uint32_t scales = smem_u32(smem + L.scales) + (uint32_t)s * kScaleBytes;
    const int row_off = warp * 32;   // first row of this warp inside the stage
    const int nrows = dead ? 0 : max(0, min(kChunk, vmax_seg - c * kChunk));

    if (warp * 32 < nrows) {
      const bool two = warp * 32 + 16 < nrows;        // the warp's second 16-row tile holds data
      const uint32_t sf_base = smem_u32(smem + L.sfl) + (uint32_t)warp * 512u;
      stage_group_scales(scales, row_off, sf_base, lane);
      // this lane's row after the reduce-scatter: rows 8t .. 8t+7 of the warp's 32 are the
      // 8-entry block t, one row per lane g
      const int r_mine = warp * 32 + 8 * t + g;
      for (int ql = 0; ql < nql; ++ql) {
        if (nql > 1) load_query_regs(ql);
        float v = score_rows32(codes, row_off, sf_base, two, B, wr, lane);
        const bool ok = c * kChunk + r_mine < svis[ql];
        v = ok ? v : -INFINITY;
        const uint32_t bin = order_key(v) >> kHistShift;
        {
          const int row = cur_seg * p.nq + ql;
          p.scores[(size_t)row * p.ld_s + c * kChunk + r_mine] = v;
          if (ok) atomicAdd(hist_sm + (2 * ql) * (kHistBins / 2) + (bin >> 1), (bin & 1) ? 0x10000u : 1u);
          // 8-entry block max: block t of the warp is held by lanes g = 0..7 of column t
          float bm = v;
          bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 4));
          bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 8));
          bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 16));
          const int jb = ((c * kChunk + warp * 32) >> 3) + t;
          if (g == 0 && jb * 8 < svis[ql]) {
            p.blkmax[(size_t)row * p.ld_b + jb] = bm;
            const uint32_t bb = order_key(bm) >> kHistShift;
            atomicAdd(hist_sm + (2 * ql + 1) * (kHistBins / 2) + (bb >> 1), (bb & 1) ? 0x10000u : 1u);
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
  if (cur_seg >= 0) finish_segment(cur_seg, seg_items);
}

// ------------------------------------------------------------------ select
constexpr int kSelThreads = 512;
constexpr int kSelSplit = 4;        // CTAs (one cluster) per (row, selection)
constexpr int kSelStage = 4096;     // candidates ranked from shared memory; more are ranked from L2
constexpr int kSelRankMax = 512;    // candidates ranked by counting up to this many

// the smallest float whose order key is `key` (inverse of order_key)
__device__ __forceinline__ float key_to_float(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

// The exact top-K of one score array (positions, or 8-position block maxima), emitted ascending,
// by one cluster of 4 CTAs, CTA r owning the quarter [r Q, (r + 1) Q) of the array:
//  1. stream the quarter once: an element whose 12-bit key bin lies above the threshold bin the
//     score pass found is taken at once (a bit in the quarter's bitmap); an element in the
//     threshold bin becomes a candidate (its index, written to the workspace). A float compare
//     against the bin's lowest value rejects most elements before any key arithmetic;
//  2. each CTA publishes (taken, candidates) counts; after one cluster barrier every CTA makes
//     the same cut among all candidates by (low key bits desc, index asc): a histogram of their
//     next 12 key bits, then a count over those left in its threshold bin (an 11-bit-digit radix
//     select when many tie in 24 key bits) - and marks its own;
//  3. each CTA emits its quarter's bitmap in ascending order at the offset the counts give
//     (blocks expanded into 8 pool positions); CTA 0 pads the tail and clears the row's histogram
//     and selection state for the next call.
__global__ void __cluster_dims__(kSelSplit, 1, 1) __launch_bounds__(kSelThreads) select_kernel(const SelectParams p) {
  extern __shared__ __align__(16) uint32_t fsm[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rank = (int)cluster_rank();
  const int unit = blockIdx.x / kSelSplit;            // (row, selection)
  const int row = unit >> 1, which = unit & 1;
  griddep_wait();
  griddep_launch_dependents();
  const int vis = (int)imin64(__ldg(p.vis + row), p.max_vis);
  const float* data;
  int n, K;
  if (which == 0) {
    data = p.scores + (size_t)row * p.ld_s;
    n = vis;
    K = kTopK;
  } else {
    data = p.blkmax + (size_t)row * p.ld_b;
    n = (vis + kBlk - 1) / kBlk;
    K = kCandBlocks;
  }
  SelState* st = p.state + 2 * row + which;
  const int Q = ((n + kSelSplit - 1) / kSelSplit + 31) & ~31;   // quarter length, a multiple of 32
  const int lo = min(n, rank * Q), hi = min(n, lo + Q);
  const int nwq = Q >> 5;                              // bitmap words of a quarter
  uint32_t* bitmap = fsm;                              // [nwq]
  uint32_t* shist = fsm + ((nwq + 3) & ~3);           // [4096] second-level bins, then radix digits
  int* scratch = reinterpret_cast<int*>(shist + kHistBins);   // [64]
  uint64_t* cst = reinterpret_cast<uint64_t*>(scratch + 64);   // [kSelStage] candidate composites
  // candidate indices of CTA c: the workspace's candidate row, split in quarters
  int* cand_row = p.cand + (size_t)row * p.ld_cand + (which ? p.ld_s : 0);
  int* xcnt = p.sure + (size_t)row * p.ld_sure + 8 * which;   // [4 CTAs][taken, candidates]

  __shared__ int s_thr, s_nvalid, s_ready, s_ncand, s_nsure;
  __shared__ int s_digit, s_above, s_cnt;
  __shared__ int s_taken[kSelSplit];
  __shared__ __align__(8) uint64_t s_cut;
  __shared__ __align__(8) uint64_t s_rk[kSelRankMax];   // candidates ranked by counting
  __shared__ int s_out[2], s_nrk;
  if (tid == 0) {
    volatile SelState* vs = st;
    s_ready = vs->ready;
    s_thr = vs->thr_bin;
    s_nvalid = vs->nvalid;
    s_ncand = 0;
    s_nsure = 0;
  }
  if (tid < kSelSplit) s_taken[tid] = 0;
  if (tid == 0) s_nrk = 0;
  for (int i = tid; i < nwq; i += kSelThreads) bitmap[i] = 0;
  __syncthreads();
  const int thr = s_ready ? s_thr : -1;
  const int Keff = min(K, s_ready ? s_nvalid : 0);

  // 1. one pass over the quarter: 8 float4 loads in flight per thread
  const float f_lo = (thr < 0) ? -INFINITY : key_to_float((uint32_t)thr << kHistShift);
  int* my_cand = cand_row + (size_t)rank * Q;
  for (int base = lo; base < hi; base += 32 * kSelThreads) {
    float4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int e0 = base + 4 * (u * kSelThreads + tid);
      v[u] = (e0 < hi) ? __ldcg(reinterpret_cast<const float4*>(data + e0))
                       : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int e0 = base + 4 * (u * kSelThreads + tid);
      const float f[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int e = e0 + j;
        if (!(f[j] >= f_lo) || f[j] == -INFINITY || e >= hi) continue;
        const uint32_t key = order_key(f[j]);
        const int bin = (int)(key >> kHistShift);
        if (thr < 0 || bin > thr) {
          atomicOr(bitmap + ((e - lo) >> 5), 1u << ((e - lo) & 31));
          atomicAdd(&s_nsure, 1);
        } else if (bin == thr) {
          my_cand[atomicAdd(&s_ncand, 1)] = e;          // at most Q per quarter
        }
      }
    }
  }
  __syncthreads();
  if (tid == 0) {
    __stcg(xcnt + 2 * rank, s_nsure);
    __stcg(xcnt + 2 * rank + 1, s_ncand);
  }
  cluster_sync_all();                 // every quarter's counts and candidates are in L2

  // 2. the cut among the candidates: candidate i is taken iff (comp & mask) >= prefix
  int sure_c[kSelSplit], cbase[kSelSplit], S = 0, C = 0;
#pragma unroll
  for (int c = 0; c < kSelSplit; ++c) {
    sure_c[c] = __ldcg(xcnt + 2 * c);
    cbase[c] = C;
    C += __ldcg(xcnt + 2 * c + 1);
    S += sure_c[c];
  }
  const int need = Keff - S;
  auto cta_of = [&](int i) {
    int c = 0;
#pragma unroll
    for (int d = 1; d < kSelSplit; ++d) c += (i >= cbase[d]) ? 1 : 0;
    return c;
  };
  // composite of candidate i (global index over the four lists): low key bits, inverted index
  auto comp_at = [&](int i) -> uint64_t {
    const int c = cta_of(i);
    const int e = __ldcg(cand_row + (size_t)c * Q + (i - cbase[c]));
    return ((uint64_t)(order_key(__ldcg(data + e)) & 0xFFFFFu) << 32) | (uint64_t)(~(uint32_t)e);
  };
  const bool none = (thr < 0) || (need <= 0);
  uint64_t prefix = none ? ~0ull : 0ull, mask = none ? ~0ull : 0ull;   // none: no composite reaches ~0
  if (!none && need < C) {
    const bool staged = C <= kSelStage;
    if (staged) {
      for (int i = tid; i < C; i += kSelThreads) cst[i] = comp_at(i);
      named_bar_sync(1, kSelThreads);
    }
    auto comp = [&](int i) -> uint64_t { return staged ? cst[i] : comp_at(i); };
    // level 2: a 4096-bin histogram of the next 12 key bits (composite bits 51..40) narrows the
    // candidates still to be ranked to those sharing 24 key bits
    for (int i = tid; i < kHistBins; i += kSelThreads) shist[i] = 0u;
    named_bar_sync(1, kSelThreads);
    for (int i = tid; i < C; i += kSelThreads) atomicAdd(shist + ((comp(i) >> 40) & 0xFFFu), 1u);
    named_bar_sync(1, kSelThreads);
    smem_threshold<kSelThreads>(shist, need, scratch, s_out, tid);
    const int thr2 = s_out[0];
    const int need_r = need - s_out[1];
    prefix = (uint64_t)thr2 << 40;
    mask = 0xFFFull << 40;
    const int C2 = (int)shist[thr2];
    if (need_r < C2 && C2 <= kSelRankMax) {
      // few left: the need_r-th largest of them by counting (composites are distinct)
      for (int i0 = warp * 32; i0 < C; i0 += kSelThreads) {
        const int i = i0 + lane;
        const uint64_t c64 = (i < C) ? comp(i) : 0ull;
        const bool in = (i < C) && (c64 & mask) == prefix;
        const int j = warp_append(in, &s_nrk, lane);
        if (in) s_rk[j] = c64;
      }
      named_bar_sync(1, kSelThreads);
      for (int i = tid; i < C2; i += kSelThreads) {
        const uint64_t ci = s_rk[i];
        int better = 0;
        for (int j = 0; j < C2; ++j) better += (s_rk[j] > ci) ? 1 : 0;
        if (better == need_r - 1) s_cut = ci;
      }
      named_bar_sync(1, kSelThreads);
      prefix = s_cut;
      mask = ~0ull;
    } else if (need_r < C2) {
      // many left (ties in 24 key bits): radix select, 11-bit digits over composite bits 39..0
      int remaining = need_r;
      const int shifts[4] = {29, 18, 7, 0};
      const int widths[4] = {11, 11, 11, 7};
      constexpr int kPerD = 2048 / kSelThreads;        // 4 digit bins per thread, high first
      for (int d = 0; d < 4; ++d) {
        const int sh = shifts[d];
        const uint32_t wm = (1u << widths[d]) - 1u;
        named_bar_sync(1, kSelThreads);
        for (int i = tid; i < 2048; i += kSelThreads) shist[i] = 0u;
        named_bar_sync(1, kSelThreads);
        for (int i = tid; i < C; i += kSelThreads) {
          const uint64_t c64 = comp(i);
          if ((c64 & mask) == prefix) atomicAdd(shist + ((c64 >> sh) & wm), 1u);
        }
        named_bar_sync(1, kSelThreads);
        const int dtop = 2048 - kPerD * (tid + 1);
        int dc[kPerD], dl = 0;
#pragma unroll
        for (int i = 0; i < kPerD; ++i) {
          dc[i] = (int)shist[dtop + kPerD - 1 - i];
          dl += dc[i];
        }
        int dtot;
        const int dex = excl_scan(dl, scratch, 1, kSelThreads, &dtot, tid);
        if (dex < remaining && dex + dl >= remaining) {
          int run = dex;
#pragma unroll
          for (int i = 0; i < kPerD; ++i) {
            if (run + dc[i] >= remaining) {
              s_digit = dtop + kPerD - 1 - i;
              s_above = run;
              s_cnt = dc[i];
              break;
            }
            run += dc[i];
          }
        }
        named_bar_sync(1, kSelThreads);
        remaining -= s_above;
        prefix |= (uint64_t)s_digit << sh;
        mask |= (uint64_t)wm << sh;
        const bool all_in = (s_cnt == remaining);
        named_bar_sync(1, kSelThreads);
        if (all_in) break;
      }
    }
  }
  if (!none) {
    // mark this quarter's taken candidates; count every CTA's
    int taken_c[kSelSplit] = {0, 0, 0, 0};
    for (int i0 = warp * 32; i0 < C; i0 += kSelThreads) {
      const int i = i0 + lane;
      const uint64_t c64 = (i < C) ? (C <= kSelStage && need < C ? cst[i] : comp_at(i)) : 0ull;
      const bool taken = (i < C) && (c64 & mask) >= prefix;
      const int c = cta_of(i);
#pragma unroll
      for (int d = 0; d < kSelSplit; ++d) taken_c[d] += __popc(__ballot_sync(0xffffffffu, taken && c == d));
      if (taken && c == rank) {
        const int e = (int)(~(uint32_t)c64) - lo;
        atomicOr(bitmap + (e >> 5), 1u << (e & 31));
      }
    }
    if (lane < kSelSplit) {
      const int v = (lane == 0) ? taken_c[0] : (lane == 1) ? taken_c[1] : (lane == 2) ? taken_c[2] : taken_c[3];
      if (v) atomicAdd(s_taken + lane, v);
    }
  }
  __syncthreads();

  // 3. ascending emission at this quarter's offset
  int off = 0;
#pragma unroll
  for (int c = 0; c < kSelSplit; ++c) off += (c < rank) ? sure_c[c] + s_taken[c] : 0;
  const int per = (nwq + kSelThreads - 1) / kSelThreads;
  const int w0 = min(nwq, tid * per), w1 = min(nwq, w0 + per);
  int cnt = 0;
  for (int i = w0; i < w1; ++i) cnt += __popc(bitmap[i]);
  int total;
  int o = off + excl_scan(cnt, scratch, 1, kSelThreads, &total, tid);
  if (which == 0) {
    int32_t* out = p.topk_out + (size_t)row * kTopK;
    for (int i = w0; i < w1; ++i) {
      uint32_t m = bitmap[i];
      while (m) {
        const int b = __ffs(m) - 1;
        m &= m - 1;
        if (o < kTopK) out[o] = lo + i * 32 + b;
        ++o;
      }
    }
    if (rank == 0)
      for (int j = Keff + tid; j < kTopK; j += kSelThreads) out[j] = -1;
  } else {
    int32_t* out = p.pool_out + (size_t)row * kPool;
    for (int i = w0; i < w1; ++i) {
      uint32_t m = bitmap[i];
      while (m) {
        const int b = __ffs(m) - 1;
        m &= m - 1;
        const int blk = lo + i * 32 + b;
        if (o < kCandBlocks) {
          int4 lo4, hi4;
          const int q0 = blk * 8;
          lo4.x = (q0 + 0 < vis) ? q0 + 0 : -1;
          lo4.y = (q0 + 1 < vis) ? q0 + 1 : -1;
          lo4.z = (q0 + 2 < vis) ? q0 + 2 : -1;
          lo4.w = (q0 + 3 < vis) ? q0 + 3 : -1;
          hi4.x = (q0 + 4 < vis) ? q0 + 4 : -1;
          hi4.y = (q0 + 5 < vis) ? q0 + 5 : -1;
          hi4.z = (q0 + 6 < vis) ? q0 + 6 : -1;
          hi4.w = (q0 + 7 < vis) ? q0 + 7 : -1;
          reinterpret_cast<int4*>(out + 8 * o)[0] = lo4;
          reinterpret_cast<int4*>(out + 8 * o)[1] = hi4;
        }
        ++o;
      }
    }
    if (rank == 0)
      for (int j = 8 * min(Keff, kCandBlocks) + tid; j < kPool; j += kSelThreads) out[j] = -1;
  }
  // clear this row's histogram and state for the next call (every CTA read the state before the
  // cluster barrier above)
  if (rank == 0) {
    uint32_t* gh = p.hist + (size_t)(2 * row + which) * kHistBins;
    for (int i = tid; i < kHistBins; i += kSelThreads) gh[i] = 0;
    if (tid == 0) {
      st->thr_bin = 0;
      st->above = 0;
      st->nvalid = 0;
      st->nsure = 0;
      st->ncand = 0;
      st->ready = 0;
    }
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
  const int64_t q = ((std::max<int64_t>(p.max_vis, 1) + kSelSplit - 1) / kSelSplit + 31) / 32;   // bitmap words of a quarter
  const size_t smem = (size_t)((q + 3) & ~3) * 4 + kHistBins * 4 + 64 * 4 + (size_t)kSelStage * 8;
  cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(select_kernel), smem);
  if (e != cudaSuccess) return e;
  // one cluster of 4 CTAs per (row, selection): the position top-512, then the block top-2048
  return launch_pdl(select_kernel, dim3((unsigned)(rows * 2 * kSelSplit)), dim3(kSelThreads), smem, s, p);
}

}  // namespace hsa
