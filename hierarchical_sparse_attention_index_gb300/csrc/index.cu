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
// Selection (exact; ties to the lower index), one CTA per (row, selection): elements above the
// threshold bin are taken, elements in it become candidates, and an 11-bit-digit radix select
// over (low key bits, inverted index) composites picks the remaining ones. A bitmap over the
// index space then emits the result in ascending order, expands blocks into the candidate
// pool, and clears the workspace state.
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
            bulk_g2s(dcodes, p.ik_q + e0 * 64, (uint32_t)nc * 64u, full);
            bulk_g2s(dscales, p.ik_s + e0 * 4, (uint32_t)nc * 4u, full);
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
constexpr int kSelThreads = 1024;
constexpr int kFinStage = 8192;   // threshold-bin candidates kept in shared memory; more spill to the workspace

// the smallest float whose order key is `key` (inverse of order_key)
__device__ __forceinline__ float key_to_float(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

__device__ __forceinline__ int block_excl_scan_1024(int v, int* scratch, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int tt = scratch[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, tt, o);
      if (lane >= o) tt += y;
    }
    scratch[lane] = tt;
  }
  __syncthreads();
  const int before = warp ? scratch[warp - 1] : 0;
  *total = scratch[31];
  __syncthreads();
  return before + x - v;
}

// One CTA per (row, selection): the exact top-K of one score array, emitted ascending.
//  1. stream the row once: an element whose 12-bit key bin lies above the threshold bin the
//     score pass found is taken at once (a bit in the index bitmap); an element in the
//     threshold bin becomes a candidate (index + low 20 key bits, in shared memory);
//  2. an 11-bit-digit radix select over the candidates' (low key bits, inverted index)
//     composites takes the remaining K - above, ties to the lower index;
//  3. the bitmap is emitted in ascending order (Reindex: through the pool; Full blocks: expanded
//     into 8 positions each), and the row's histogram and state are cleared for the next call.
__global__ void __launch_bounds__(kSelThreads) select_kernel(const SelectParams p) {
  extern __shared__ __align__(16) uint32_t fsm[];
  const int row = blockIdx.x, which = blockIdx.y;
  const int tid = threadIdx.x;
  griddep_wait();
  griddep_launch_dependents();
  const int vis = (int)imin64(__ldg(p.vis + row), p.max_vis);
  const float* data;
  int n, K;
  int64_t cand_off = 0;
  if (which == 0) {
    data = p.scores + (size_t)row * p.ld_s;
    n = vis;
    K = kTopK;
  } else {
    data = p.blkmax + (size_t)row * p.ld_b;
    n = (vis + kBlk - 1) / kBlk;
    K = kCandBlocks;
    cand_off = p.ld_s;
  }
  SelState* st = p.state + 2 * row + which;
  const int nwords = (max(n, 1) + 31) >> 5;
  uint32_t* bitmap = fsm;                       // [nwords]
  uint32_t* shist = fsm + ((nwords + 3) & ~3);  // [2048]
  int* scratch = reinterpret_cast<int*>(shist + 2048);   // [64]
  int* s_cidx = scratch + 64;                   // [kFinStage]
  uint32_t* s_ckey = reinterpret_cast<uint32_t*>(s_cidx + kFinStage);   // [kFinStage]
  int* gcand = p.cand + (size_t)row * p.ld_cand + cand_off;              // overflow candidates
  const int gcap = (int)(which == 0 ? p.ld_s : p.ld_b);

  __shared__ int s_thr, s_nvalid, s_ready, s_ncand, s_nsure;
  __shared__ int s_digit, s_above, s_cnt;
  if (tid == 0) {
    volatile SelState* vs = st;
    s_ready = vs->ready;
    s_thr = vs->thr_bin;
    s_nvalid = vs->nvalid;
    s_ncand = 0;
    s_nsure = 0;
  }
  for (int i = tid; i < nwords; i += kSelThreads) bitmap[i] = 0;
  __syncthreads();
  const int thr = s_ready ? s_thr : -1;
  const int Keff = min(K, s_ready ? s_nvalid : 0);

  // 1. one pass over the row: 8 float4 loads in flight per thread; one float compare against the
  //    lowest value of the threshold bin rejects most elements before any key arithmetic (it is
  //    conservative: the bin test below is exact)
  const float f_lo = (thr < 0) ? -INFINITY : key_to_float((uint32_t)thr << kHistShift);
  const int n4 = (n + 3) >> 2;
  for (int base = 0; base < n4; base += 8 * kSelThreads) {
    float4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i4 = base + u * kSelThreads + tid;
      v[u] = (i4 < n4) ? __ldcg(reinterpret_cast<const float4*>(data) + i4)
                       : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int e0 = 4 * (base + u * kSelThreads + tid);
      const float f[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int e = e0 + j;
        if (!(f[j] >= f_lo) || f[j] == -INFINITY || e >= n) continue;
        const uint32_t key = order_key(f[j]);
        const int bin = (int)(key >> kHistShift);
        if (thr < 0 || bin > thr) {
          atomicOr(bitmap + (e >> 5), 1u << (e & 31));
          atomicAdd(&s_nsure, 1);
        } else if (bin == thr) {
          const int slot = atomicAdd(&s_ncand, 1);
          if (slot < kFinStage) {
            s_cidx[slot] = e;
            s_ckey[slot] = key & 0xFFFFFu;
          } else if (slot - kFinStage < gcap) {
            gcand[slot - kFinStage] = e;
          } else {
            flag_status(p.status, HSA_FLAG_INDEX_RANGE);
          }
        }
      }
    }
  }
  __syncthreads();
  const int ncand = min(s_ncand, kFinStage + gcap);
  const int need = Keff - s_nsure;

  // 2. exact selection of the remaining `need` among the candidates
  if (thr >= 0 && need > 0 && ncand > 0) {
    auto comp_of = [&](int i) -> uint64_t {
      int e;
      uint32_t k20;
      if (i < kFinStage) {
        e = s_cidx[i];
        k20 = s_ckey[i];
      } else {
        e = __ldcg(gcand + (i - kFinStage));
        k20 = order_key(__ldcg(data + e)) & 0xFFFFFu;
      }
      return ((uint64_t)k20 << 32) | (uint64_t)(~(uint32_t)e);
    };
    uint64_t prefix = 0, mask = 0;
    int remaining = need;
    const int shifts[5] = {41, 30, 19, 8, 0};
    const int widths[5] = {11, 11, 11, 11, 8};
    for (int d = 0; d < 5; ++d) {
      const int sh = shifts[d];
      const uint32_t wm = (1u << widths[d]) - 1u;
      for (int i = tid; i < 2048; i += kSelThreads) shist[i] = 0;
      __syncthreads();
      for (int i = tid; i < ncand; i += kSelThreads) {
        const uint64_t comp = comp_of(i);
        if ((comp & mask) == prefix) atomicAdd(shist + ((comp >> sh) & wm), 1u);
      }
      __syncthreads();
      // 2048 bins, 2 per thread, highest first
      const int hi_bin = 2047 - 2 * tid;
      const int c_hi = (int)shist[hi_bin], c_lo = (int)shist[hi_bin - 1];
      int tot;
      const int excl = block_excl_scan_1024(c_hi + c_lo, scratch, &tot);
      if (excl < remaining && excl + c_hi + c_lo >= remaining) {
        if (excl + c_hi >= remaining) {
          s_digit = hi_bin;
          s_above = excl;
          s_cnt = c_hi;
        } else {
          s_digit = hi_bin - 1;
          s_above = excl + c_hi;
          s_cnt = c_lo;
        }
      }
      __syncthreads();
      remaining -= s_above;
      prefix |= (uint64_t)s_digit << sh;
      mask |= (uint64_t)wm << sh;
      const bool all_in = (s_cnt == remaining);
      __syncthreads();
      if (all_in) break;
    }
    for (int i = tid; i < ncand; i += kSelThreads) {
      const uint64_t comp = comp_of(i);
      if ((comp & mask) >= prefix) {
        const int e = (int)(~(uint32_t)(comp & 0xFFFFFFFFull));
        atomicOr(bitmap + (e >> 5), 1u << (e & 31));
      }
    }
  }
  __syncthreads();

  // 3. ascending emission
  const int per = (nwords + kSelThreads - 1) / kSelThreads;
  const int w0 = min(nwords, tid * per), w1 = min(nwords, w0 + per);
  int cnt = 0;
  for (int i = w0; i < w1; ++i) cnt += __popc(bitmap[i]);
  int total;
  int o = block_excl_scan_1024(cnt, scratch, &total);
  if (which == 0) {
    int32_t* out = p.topk_out + (size_t)row * kTopK;
    for (int i = w0; i < w1; ++i) {
      uint32_t m = bitmap[i];
      while (m) {
        const int b = __ffs(m) - 1;
        m &= m - 1;
        if (o < kTopK) out[o] = i * 32 + b;
        ++o;
      }
    }
    for (int j = total + tid; j < kTopK; j += kSelThreads) out[j] = -1;
  } else {
    int32_t* out = p.pool_out + (size_t)row * kPool;
    for (int i = w0; i < w1; ++i) {
      uint32_t m = bitmap[i];
      while (m) {
        const int b = __ffs(m) - 1;
        m &= m - 1;
        const int blk = i * 32 + b;
        if (o < kCandBlocks) {
          int4 lo, hi;
          const int q0 = blk * 8;
          lo.x = (q0 + 0 < vis) ? q0 + 0 : -1;
          lo.y = (q0 + 1 < vis) ? q0 + 1 : -1;
          lo.z = (q0 + 2 < vis) ? q0 + 2 : -1;
          lo.w = (q0 + 3 < vis) ? q0 + 3 : -1;
          hi.x = (q0 + 4 < vis) ? q0 + 4 : -1;
          hi.y = (q0 + 5 < vis) ? q0 + 5 : -1;
          hi.z = (q0 + 6 < vis) ? q0 + 6 : -1;
          hi.w = (q0 + 7 < vis) ? q0 + 7 : -1;
          reinterpret_cast<int4*>(out + 8 * o)[0] = lo;
          reinterpret_cast<int4*>(out + 8 * o)[1] = hi;
        }
        ++o;
      }
    }
    for (int j = 8 * min(total, kCandBlocks) + tid; j < kPool; j += kSelThreads) out[j] = -1;
  }
  // clear this row's histogram and state for the next call
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

}  // namespace

template <bool kOneQuery>
cudaError_t launch_scan_variant(const ScanParams& p, int num_sms, cudaStream_t s) {
  const ScanSmemLayout L = scan_smem_layout(p.nq);
  auto kern = index_scan_kernel<kOneQuery>;
  static int set_bytes = 0;        // the attribute is per function, set to the largest size seen
  if ((int)L.total > set_bytes) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.total);
    if (e != cudaSuccess) return e;
    set_bytes = (int)L.total;
  }
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
  const int nsel = 2;               // position top-512 and block top-2048
  const int64_t nwords = (std::max<int64_t>(p.max_vis, 1) + 31) / 32;
  const size_t smem = (size_t)((nwords + 3) & ~3) * 4 + 2048 * 4 + 64 * 4 + (size_t)kFinStage * 8;
  static size_t set_bytes = 0;
  if (smem > set_bytes) {
    cudaError_t e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    set_bytes = smem;
  }
  return launch_pdl(select_kernel, dim3((unsigned)rows, (unsigned)nsel), dim3(kSelThreads), smem, s, p);
}

}  // namespace hsa
