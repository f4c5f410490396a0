// Fused Reindex indexer ([CED] Figure 5 right: the Reindex pass rescored over the candidate pool;
// [ARCH] §3.3 候选池 重排; [10100] 层次化稀疏索引器): per (request, query) row, score the
// 16,384 pool slots s = sum_h w_h ReLU(q_h . k) and emit the exact top-512 (ties to the lower
// slot), ascending, in one launch.
//
// One thread-block cluster of 4 CTAs per row; CTA r owns slots [4096 r, 4096 r + 4096) (with
// the window tail, CTA 3 also owns the 160 slots past 16,384, scored as a 9th group by its warps
// 0..4, so the slot order stays the position order):
//  1. 16 warps score 256 slots each: 8 groups of 32 slots (four 8-entry runs) gathered with
//     cp.async into a per-warp ring 4 groups ahead, scored with warp MMAs (shared with the scan
//     kernel); scores stay in shared memory with a 4096-bin histogram of their top 12 key bits;
//  2. the CTA finds its own threshold bin b_r (the bin of its 512-th largest key) and lists, in
//     its own shared memory, every valid element in a bin >= b_r (order key and slot), with the
//     list's count and its number of valid elements. The row's top-512 lies inside the union of
//     the four lists: an element of CTA r in the row's top-512 is in CTA r's own top-512;
//  3. after one cluster barrier every CTA reads the four lists over distributed shared memory
//     (a split cluster arrive/wait keeps each CTA alive until its peers are done) and selects
//     the same top-K,
//     K = min(512, valid elements of the row): a histogram of the union's top key bits gives the
//     threshold bin, and the elements in it are ranked by (key desc, slot asc) - by counting
//     when there are few, by an exact radix select otherwise;
//  4. each CTA writes its selected slots' positions in ascending slot order at the offset given
//     by the counts of the CTAs before it; CTA 0 pads the tail with -1.
#include "hsa_common.cuh"
#include "hsa_hist.cuh"
#include "hsa_internal.h"
#include "hsa_score.cuh"

namespace hsa {
namespace {

constexpr int kRxWarps = 16;
constexpr int kRxThreads = kRxWarps * 32;
constexpr int kRxCluster = kRxSplit;
constexpr int kSlotsPerCta = kPool / kRxCluster;          // 4096
constexpr int kSlotsPerWarp = kSlotsPerCta / kRxWarps;    // 256
constexpr int kGroups = kSlotsPerWarp / 32;               // 8 groups of 32 slots per warp
constexpr int kRxRing = 5;                                // gathers run 4 groups ahead
constexpr uint32_t kGrpCodes = 32 * 64, kGrpScales = 32 * 4;
constexpr int kRankMax = 512;                             // threshold-bin elements ranked by counting up to this many
constexpr int kPerT = kHistBins / kRxThreads;             // 8 bins (or slots) per thread
constexpr int kTail = HSA_POOL_TAIL_SLOTS;                // slots past kPool with the window tail (CTA 3)
constexpr int kTailGroups = kTail / 32;                   // 5 groups of 32: warps 0..4 of CTA 3
constexpr int kLocMax = kSlotsPerCta + kTail;             // local slots of CTA 3 with the tail

// shared-memory layout (bytes)
constexpr uint32_t kOffRing = 0;                                                  // [16 warps][5][codes|scales]
constexpr uint32_t kRingBytes = (uint32_t)kRxWarps * kRxRing * (kGrpCodes + kGrpScales);
constexpr uint32_t kOffSlots = kOffRing + kRingBytes;                             // [16][5][32] int
constexpr uint32_t kOffBfrag = kOffSlots + kRxWarps * kRxRing * 32 * 4;
constexpr uint32_t kOffWsc = kOffBfrag + kQFragWords * 4;
constexpr uint32_t kOffSfl = kOffWsc + kQWeights * 4;                              // [16 warps][512 B]
constexpr uint32_t kOffSc = kOffSfl + kRxWarps * 512;                              // [4256] scores
constexpr uint32_t kOffHist = kOffSc + kLocMax * 4;                                // [4096] counts
constexpr uint32_t kOffSel = kOffHist + kHistBins * 4;                             // [4256 bits] taken slots
constexpr uint32_t kSelBytes = (kLocMax / 8 + 15) / 16 * 16;                     // bitmap bytes, 16-aligned
constexpr uint32_t kOffScr = kOffSel + kSelBytes;                                  // scratch ints
constexpr uint32_t kScrInts = 128;
constexpr uint32_t kRxSmem = kOffScr + kScrInts * 4;
static_assert(kRxSmem <= 232448, "shared memory");
// after scoring, the rings hold the union (64-bit composites) and the score array the ranked
// threshold-bin elements
static_assert((uint32_t)(kPool + kTail) * 8 + kLocMax * 8 <= kRingBytes, "union staging and own list fit the rings");
static_assert(kTail % 32 == 0 && kTailGroups <= kRxWarps, "tail groups");
// scr + 84 holds a 64-bit composite: every region starts 16-byte aligned
static_assert(kOffSc % 16 == 0 && kOffHist % 16 == 0 && kOffSel % 16 == 0 && kOffScr % 16 == 0, "alignment");
static_assert(kRankMax * 8 <= kSlotsPerCta * 4, "ranked elements fit the score array");

// (order key, inverted row slot): larger = better, ties to the lower slot
__device__ __forceinline__ uint64_t comp_of(uint32_t key, uint32_t row_slot) {
  return ((uint64_t)key << 32) | (uint64_t)(~row_slot);
}
__device__ __forceinline__ uint32_t slot_of(uint64_t comp) { return ~(uint32_t)comp; }
__device__ __forceinline__ int bin_of(uint64_t comp) { return (int)(comp >> (32 + kHistShift)); }

// Threshold bin of a top-K over `hist` into scr[64], scr[65] (smem_threshold over this CTA's threads)
__device__ __forceinline__ int find_threshold(const uint32_t* hist, int K, int* scr, int tid) {
  return smem_threshold<kRxThreads>(hist, K, scr, scr + 64, tid);
}

template <bool kPoolTail>
__global__ void __cluster_dims__(kRxCluster, 1, 1) __launch_bounds__(kRxThreads, 1)
    reindex_kernel(const ReindexParams p) {
  extern __shared__ __align__(1024) uint8_t rsm[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rank = (int)cluster_rank();
  const int row = blockIdx.x / kRxCluster;
  uint32_t* hist = reinterpret_cast<uint32_t*>(rsm + kOffHist);
  float* sc = reinterpret_cast<float*>(rsm + kOffSc);
  uint32_t* sel = reinterpret_cast<uint32_t*>(rsm + kOffSel);
  int* scr = reinterpret_cast<int*>(rsm + kOffScr);
  uint32_t* bfrag = reinterpret_cast<uint32_t*>(rsm + kOffBfrag);
  float* wsc = reinterpret_cast<float*>(rsm + kOffWsc);

  for (int i = tid; i < kHistBins; i += kRxThreads) hist[i] = 0u;
  for (int i = tid; i < kLocMax / 32; i += kRxThreads) sel[i] = 0u;
  if (tid < kScrInts) scr[tid] = 0;
  // Inside schedule_step everything this kernel reads was complete before it was launched (the
  // pool two or more kernels earlier, q, w and vis before the step), so it scores while the
  // previous kernel drains and waits for it only before its first global write. The next
  // kernel is released after the scoring, whose gathers it would otherwise slow down.
  if (!p.inputs_ready) griddep_wait();

  const int vis = __ldg(p.vis + row);
  const int32_t* pool_row = p.pool + (size_t)row * p.pool_ld;
  const bool has_tail = kPoolTail && rank == kRxCluster - 1;

  // ---------------------------------------------------------------- 1. score this warp's 256 slots
  const int slot0 = kSlotsPerCta * rank + kSlotsPerWarp * warp;   // first slot (row-relative) of the warp
  // group g < 8: the warp's own slots; group 8 (CTA 3's warps 0..4 with the tail): slots
  // kPool + 32 warp .. + 31, local kSlotsPerCta + 32 warp
  const int ngroups = kGroups + ((has_tail && warp < kTailGroups) ? 1 : 0);
  const int64_t ebase = (int64_t)(row / p.nq) * p.cap;
  const uint32_t ring = smem_u32(rsm + kOffRing) + (uint32_t)(warp * kRxRing) * (kGrpCodes + kGrpScales);
  int* slots = reinterpret_cast<int*>(rsm + kOffSlots) + warp * kRxRing * 32;
  // a group's pool values are loaded one gather ahead, so a gather never waits for them. The
  // pool is another kernel's output: coherent loads only (see griddep_wait)
  auto pool_val = [&](int grp) {
    if (grp >= ngroups) return -1;
    return __ldcg(pool_row + (grp < kGroups ? slot0 + 32 * grp : kPool + 32 * warp) + lane);
  };
  auto gather = [&](int grp, int pv) {
    const int rs = grp % kRxRing;
    const uint32_t dc = ring + (uint32_t)rs * (kGrpCodes + kGrpScales);
    gather_runs<kPoolTail>(p.ik_q, p.ik_s, ebase, p.cap, vis, pv, lane, dc, dc + kGrpCodes, slots + rs * 32, p.status);
  };
  {
    // the prologue's pool values go in flight before the query is staged
    int pv0[kRxRing - 1];
#pragma unroll
    for (int k = 0; k < kRxRing - 1; ++k) pv0[k] = pool_val(k);
    if (tid < 256) stage_query(p.q + (size_t)row * kHIdx * kDIdx, p.w + (size_t)row * kHIdx, bfrag, wsc, tid);
#pragma unroll
    for (int k = 0; k < kRxRing - 1; ++k) gather(k, pv0[k]);
  }
  int pv_next = pool_val(kRxRing - 1);
  __syncthreads();                    // staged query visible
  uint32_t B[2][8][2];
  float wr[2][2];
  load_query_frags(bfrag, wsc, lane, B, wr);
  const uint32_t sf_base = smem_u32(rsm + kOffSfl) + (uint32_t)warp * 512u;
  const int g = lane >> 2, t = lane & 3;
#pragma unroll 1
  for (int k = 0; k < ngroups; ++k) {
    if (k + kRxRing - 1 < ngroups) {
      gather(k + kRxRing - 1, pv_next);
      pv_next = pool_val(k + kRxRing);
    } else {
      cp_async_commit();
    }
    cp_async_wait<kRxRing - 1>();     // group k's runs have landed
    __syncwarp();
    const int rs = k % kRxRing;
    const uint32_t codes = ring + (uint32_t)rs * (kGrpCodes + kGrpScales);
    stage_group_scales(codes + kGrpCodes, 0, sf_base, lane);
    float v = score_rows32(codes, 0, sf_base, B, wr, lane);
    const bool ok = slots[rs * 32 + 8 * t + g] >= 0;
    v = ok ? v : -INFINITY;
    const int ls = (k < kGroups ? kSlotsPerWarp * warp + 32 * k : kSlotsPerCta + 32 * warp) + 8 * t + g;   // CTA-local slot
    sc[ls] = v;
    if (ok) atomicAdd(hist + (order_key(v) >> kHistShift), 1u);
    __syncwarp();                     // ring buffer rs is free for the gather 4 groups ahead
  }
  __syncthreads();

  griddep_launch_dependents();
  if (p.inputs_ready) griddep_wait();
  // ---------------------------------------------------------------- 2. publish this CTA's own top region
  // scr: [0, 32) scan scratch; 64, 65 threshold bin and count above it; 72 published count;
  // 73 ranked count; 76 + c slots CTA c keeps; 80..82 radix digit, count above it, count in it;
  // 84..85 the cut composite of the rank count
  const int nval_local = find_threshold(hist, kTopK, scr, tid);
  const int lthr = scr[64];
  // This CTA's list stays in its own shared memory (the rings are free now): entries at lst,
  // the count and the number of valid elements at scr[90], scr[91]; the peers read them over
  // distributed shared memory after the cluster barrier. The union is staged at ust.
  uint64_t* ust = reinterpret_cast<uint64_t*>(rsm + kOffRing);
  uint64_t* lst = reinterpret_cast<uint64_t*>(rsm + kOffRing + (kPool + kTail) * 8);
  {
    // the warp's 8 rounds of appends take one atomic: round i's lanes follow rounds 0..i-1
    uint32_t keys[kPerT], bal[kPerT];
    int n = 0;
#pragma unroll
    for (int i = 0; i < kPerT; ++i) {
      const float v = sc[kPerT * tid + i];
      keys[i] = order_key(v);
      bal[i] = __ballot_sync(0xffffffffu, (v != -INFINITY) && (int)(keys[i] >> kHistShift) >= lthr);
      n += __popc(bal[i]);
    }
    int base = 0;
    if (lane == 0 && n) base = atomicAdd(scr + 72, n);
    base = __shfl_sync(0xffffffffu, base, 0);
    const uint32_t lt = (1u << lane) - 1u;
#pragma unroll
    for (int i = 0; i < kPerT; ++i) {
      if ((bal[i] >> lane) & 1u)
        lst[base + __popc(bal[i] & lt)] = comp_of(keys[i], (uint32_t)(kSlotsPerCta * rank + kPerT * tid + i));
      base += __popc(bal[i]);
    }
  }
  if (has_tail) {
    // CTA 3's tail slots kSlotsPerCta + tid, tid < 160
    const float v = (tid < kTail) ? sc[kSlotsPerCta + tid] : -INFINITY;
    const uint32_t key = order_key(v);
    const bool in = (v != -INFINITY) && (int)(key >> kHistShift) >= lthr;
    const int j = warp_append(in, scr + 72, lane);
    if (in) lst[j] = comp_of(key, (uint32_t)(kSlotsPerCta * rank + kSlotsPerCta + tid));
  }
  for (int i = tid; i < kHistBins; i += kRxThreads) hist[i] = 0u;   // read by find_threshold above
  named_bar_sync(1, kRxThreads);
  if (tid == 0) {
    scr[90] = scr[72];
    scr[91] = nval_local;
  }
  cluster_sync_all();                  // the four lists are published

  // ---------------------------------------------------------------- 3. the row's top-K over the union
  int cnt[kRxCluster], nv[kRxCluster];
  uint32_t lst_c[kRxCluster];
#pragma unroll
  for (int c = 0; c < kRxCluster; ++c) {
    const uint32_t scr_c = cluster_map(smem_u32(scr + 90), (uint32_t)c);
    cnt[c] = ld_cluster_s32(scr_c);
    nv[c] = ld_cluster_s32(scr_c + 4u);
    lst_c[c] = cluster_map(smem_u32(lst), (uint32_t)c);
  }
  int ubase[kRxCluster], U = 0, nvalid = 0;
#pragma unroll
  for (int c = 0; c < kRxCluster; ++c) {
    ubase[c] = U;
    U += cnt[c];
    nvalid += nv[c];
  }
  const int K = min(kTopK, nvalid);
  auto cta_of = [&](int i) {
    int c = 0;
#pragma unroll
    for (int d = 1; d < kRxCluster; ++d) c += (i >= ubase[d]) ? 1 : 0;
    return c;
  };
  // thread tid stages union entries tid, tid + 512, ...: a round issues all eight of its remote
  // loads before it uses any, so their latencies overlap
  constexpr int kUnionRound = 8;
  for (int i0 = 0; i0 < U; i0 += kUnionRound * kRxThreads) {
    uint64_t v[kUnionRound];
#pragma unroll
    for (int k = 0; k < kUnionRound; ++k) {
      const int i = i0 + k * kRxThreads + tid;
      if (i < U) {
        const int c = cta_of(i);
        uint32_t at = lst_c[0] + 8u * (uint32_t)(i - ubase[0]);
#pragma unroll
        for (int d = 1; d < kRxCluster; ++d)
          if (c == d) at = lst_c[d] + 8u * (uint32_t)(i - ubase[d]);
        v[k] = ld_cluster_u64(at);
      }
    }
#pragma unroll
    for (int k = 0; k < kUnionRound; ++k) {
      const int i = i0 + k * kRxThreads + tid;
      if (i < U) {
        ust[i] = v[k];
        atomicAdd(hist + bin_of(v[k]), 1u);
      }
    }
  }
  cluster_arrive();                   // done with the peers' lists (waited for before exit)
  named_bar_sync(1, kRxThreads);
  find_threshold(hist, K, scr, tid);
  const int thr = scr[64], need = K - scr[65];
  // The cut: an element is taken iff (comp & mask) >= prefix. Inside the threshold bin, a second
  // 4096-bin histogram over the next 12 key bits narrows the elements still to be ranked to those
  // sharing 24 key bits; they are ranked by counting when there are few, by an exact radix
  // select over the remaining composite bits (key bits 7..0, then the inverted slot) otherwise.
  uint64_t prefix = 0, mask = 0;
  if (thr >= 0 && need < (int)hist[thr]) {
    int need_r = need;
    prefix = (uint64_t)thr << 52;
    mask = 0xFFFull << 52;
    named_bar_sync(1, kRxThreads);    // hist[thr] read everywhere
    for (int i = tid; i < kHistBins; i += kRxThreads) hist[i] = 0u;
    named_bar_sync(1, kRxThreads);
    for (int i = tid; i < U; i += kRxThreads) {
      const uint64_t comp = ust[i];
      if ((comp & mask) == prefix) atomicAdd(hist + ((comp >> 40) & 0xFFFu), 1u);
    }
    named_bar_sync(1, kRxThreads);
    find_threshold(hist, need_r, scr, tid);
    const int thr2 = scr[64];
    need_r -= scr[65];
    prefix |= (uint64_t)thr2 << 40;
    mask |= 0xFFFull << 40;
    const int Cn2 = (int)hist[thr2];
    if (need_r < Cn2 && Cn2 <= kRankMax) {
      // few left: the need_r-th largest of them by counting
      uint64_t* rk = reinterpret_cast<uint64_t*>(sc);             // the scores are published
      for (int i0 = warp * 32; i0 < U; i0 += kRxThreads) {
        const int i = i0 + lane;
        const uint64_t comp = (i < U) ? ust[i] : 0ull;
        const bool in = (i < U) && (comp & mask) == prefix;
        const int j = warp_append(in, scr + 73, lane);
        if (in) rk[j] = comp;
      }
      named_bar_sync(1, kRxThreads);
      for (int i = tid; i < Cn2; i += kRxThreads) {
        const uint64_t ci = rk[i];
        int better = 0;
        for (int j = 0; j < Cn2; ++j) better += (rk[j] > ci) ? 1 : 0;
        if (better == need_r - 1) *reinterpret_cast<uint64_t*>(scr + 84) = ci;
      }
      named_bar_sync(1, kRxThreads);
      prefix = *reinterpret_cast<const uint64_t*>(scr + 84);
      mask = ~0ull;
    } else if (need_r < Cn2) {
      // many left (ties in 24 key bits): exact radix select, 11-bit digits over composite bits 39..0
      int remaining = need_r;
      const int shifts[4] = {29, 18, 7, 0};
      const int widths[4] = {11, 11, 11, 7};
      constexpr int kDigitBins = 2048, kPerD = kDigitBins / kRxThreads;   // 4 bins per thread, high first
      for (int d = 0; d < 4; ++d) {
        const int sh = shifts[d];
        const uint32_t wm = (1u << widths[d]) - 1u;
        named_bar_sync(1, kRxThreads);
        for (int i = tid; i < kDigitBins; i += kRxThreads) hist[i] = 0u;
        named_bar_sync(1, kRxThreads);
        for (int i = tid; i < U; i += kRxThreads) {
          const uint64_t comp = ust[i];
          if ((comp & mask) == prefix) atomicAdd(hist + ((comp >> sh) & wm), 1u);
        }
        named_bar_sync(1, kRxThreads);
        const int dtop = kDigitBins - kPerD * (tid + 1);
        int dc[kPerD], dl = 0;
#pragma unroll
        for (int i = 0; i < kPerD; ++i) {
          dc[i] = (int)hist[dtop + kPerD - 1 - i];
          dl += dc[i];
        }
        int dtot;
        const int dex = excl_scan(dl, scr, 1, kRxThreads, &dtot, tid);
        if (dex < remaining && dex + dl >= remaining) {
          int run = dex;
#pragma unroll
          for (int i = 0; i < kPerD; ++i) {
            if (run + dc[i] >= remaining) {
              scr[80] = dtop + kPerD - 1 - i;
              scr[81] = run;
              scr[82] = dc[i];
              break;
            }
            run += dc[i];
          }
        }
        named_bar_sync(1, kRxThreads);
        remaining -= scr[81];
        prefix |= (uint64_t)scr[80] << sh;
        mask |= (uint64_t)wm << sh;
        const bool all_in = (scr[82] == remaining);
        named_bar_sync(1, kRxThreads);
        if (all_in) break;
      }
    }
  } else if (thr >= 0) {
    prefix = (uint64_t)thr << 52;     // every element of the threshold bin is taken
    mask = 0xFFFull << 52;
  }
  {
    int taken_c[kRxCluster] = {0, 0, 0, 0};   // per CTA, taken elements seen by this warp
    for (int i0 = warp * 32; i0 < U; i0 += kRxThreads) {
      const int i = i0 + lane;
      const uint64_t comp = (i < U) ? ust[i] : 0ull;
      const bool taken = (i < U) && (comp & mask) >= prefix;
      const int c = cta_of(i);
#pragma unroll
      for (int d = 0; d < kRxCluster; ++d) taken_c[d] += __popc(__ballot_sync(0xffffffffu, taken && c == d));
      if (taken && c == rank) {
        const int ls = (int)slot_of(comp) - kSlotsPerCta * rank;
        atomicOr(sel + (ls >> 5), 1u << (ls & 31));
      }
    }
    if (lane < kRxCluster) {
      const int v = (lane == 0) ? taken_c[0] : (lane == 1) ? taken_c[1] : (lane == 2) ? taken_c[2] : taken_c[3];
      if (v) atomicAdd(scr + 76 + lane, v);
    }
  }
  named_bar_sync(1, kRxThreads);

  // ---------------------------------------------------------------- 4. emit this CTA's slots, ascending
  int off = 0;
#pragma unroll
  for (int c = 0; c < kRxCluster; ++c) off += (c < rank) ? scr[76 + c] : 0;
  uint32_t mine = (sel[tid >> 2] >> (kPerT * (tid & 3))) & 0xFFu;   // local slots 8 tid .. 8 tid + 7
  int total;
  int at = off + excl_scan(__popc(mine), scr, 1, kRxThreads, &total, tid);
  int32_t* out = p.topk_out + (size_t)row * kTopK;
  const int32_t* pl = pool_row + kSlotsPerCta * rank + kPerT * tid;
  while (mine) {
    const int i = __ffs(mine) - 1;
    mine &= mine - 1u;
    if (at < kTopK) out[at] = __ldcg(pl + i);
    ++at;
  }
  if (has_tail) {
    // the tail slots follow the CTA's main slots: local kSlotsPerCta + 8 tid .. + 7, tid < 20
    uint32_t mt = (tid < kTail / 8) ? (sel[kSlotsPerCta / 32 + (tid >> 2)] >> (kPerT * (tid & 3))) & 0xFFu : 0u;
    int tt;
    int at2 = off + total + excl_scan(__popc(mt), scr, 1, kRxThreads, &tt, tid);
    const int32_t* plt = pool_row + kPool + kPerT * tid;
    while (mt) {
      const int i = __ffs(mt) - 1;
      mt &= mt - 1u;
      if (at2 < kTopK) out[at2] = __ldcg(plt + i);
      ++at2;
    }
  }
  if (rank == 0)
    for (int j = K + tid; j < kTopK; j += kRxThreads) out[j] = -1;
  cluster_wait();                     // no peer still reads this CTA's list
}

}  // namespace

cudaError_t launch_reindex(const ReindexParams& p, cudaStream_t s) {
  auto kern = p.tail ? reindex_kernel<true> : reindex_kernel<false>;
  cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(kern), kRxSmem);
  if (e != cudaSuccess) return e;
  const int rows = p.batch * p.nq;
  return launch_pdl(kern, dim3(rows * kRxCluster), dim3(kRxThreads), kRxSmem, s, p);
}

}  // namespace hsa
