// Sparse attention over the selected FP4 main-KV rows plus the FP8 SWA tail
// ([CED] Figure 4: Selected Main KV ⊕ SWA KV -> Core Attention; [890B] 注意力实际有多稀:
// 512 + 128 = 640 positions; [ARCH] §7: dequantise before attention, no FP4 matmul needed).
//
// One thread-block cluster of 4 CTAs per (request, query). CTA j owns 160 keys: top-k slots
// [128j, 128j+128) and SWA window rows [32j, 32j+32). Four CTAs per row fit a batch of 32
// requests in one wave of 128 SMs. Each CTA runs 16 worker warps and one MMA warp:
//  1. the 64x512 bf16 query arrives by TMA (each CTA loads all of it into its own shared
//     memory), already in the 128B-swizzled K-major layout. The workers
//     issue the row loads (the 160 rows, gathered once and shared by all 64 heads), convert
//     the query in place to f16 after a per-head power-of-two shift (exact within f16; each
//     warp owns 4 whole heads, so no block barrier), and dequantise the rows to f16
//     (E2M1 x scale, or E4M3 for SWA) into a 128B-swizzled K-major tile, 128 dims at a time;
//  2. the MMA warp runs S = Q . K^T on tcgen05 as M = 64 heads by N = 160 keys (TMEM
//     accumulators), each 128-dim step as soon as all workers have converted it. The tensor
//     core takes 2 N-columns per clock whatever M is, so this costs 32 x 80 clocks, against
//     64 x 48 (shared-memory bound) for S^T in two M = 128, N = 64 passes;
//  3. the workers run a softmax local to the 160 keys (own max m_c and sum l_c per head): in
//     the M = 64 accumulator layout each head is one TMEM lane, so a thread holds 40 of its
//     head's logits and four warps merge (max, sum) through shared memory. P (f16) is written
//     as the next B operand; no cluster exchange is needed before PV;
//  4. the MMA warp runs O^T[512 dims][64 heads] = V^T . P^T, reading the same tile as an
//     MN-major A operand (K = V = the 512-d latent), one 128-dim M-tile at a time;
//  5. each worker drains one output dimension of a finished M-tile, normalised by l_c: the 48
//     heads the other CTAs combine go to the workspace (L2) as f16, 8 heads per 16-byte unit
//     (a warp stores 32 consecutive dimensions of a unit: 512 contiguous bytes), this CTA's own
//     16 stay in registers in fp32. (m_c, l_c) of the 16 heads a peer owns go straight into the
//     peer's shared memory before PV (cluster barrier phase A), the partials after (phase B);
//     each CTA then forms its 16 heads as sum_c w_c (O_c / l_c), w_c = exp(m_c - M) l_c /
//     sum_c' exp(m_c' - M) l_c', over c in rank order (deterministic). L2 moves the partials
//     several times faster than distributed shared memory; the normalised partial is a convex
//     combination of f16 tile values, so it cannot leave the f16 range.
// Setup (TMEM allocation, barrier init, the arrive half of a cluster barrier whose wait comes
// before the first store into a peer's shared memory) runs before the programmatic-dependency
// wait, so it overlaps the tail of the previous kernel in the stream. Every wait is bounded.
#include "hsa_common.cuh"
#include "hsa_internal.h"
#include "hsa_tc.cuh"

namespace hsa {
namespace {

constexpr int kWorkWarps = 16;                           // load, convert, softmax, drain, combine
constexpr int kWorkThreads = kWorkWarps * 32;
constexpr int kAttnThreads = kWorkThreads + 32;          // + one warp that issues the tcgen05 MMAs
constexpr int kCluster = kAttnSplit;
constexpr int kRows = 160;                               // keys per CTA
constexpr int kTopRows = 128;
constexpr uint32_t kKbStride = kRows * 128u;             // bytes per 64-dim block of the tile
constexpr uint32_t kTileBytes = 8 * kKbStride;           // 160 KB f16 tile
constexpr uint32_t kQBytes = kHAtt * kDLat * 2;          // 64 KB f16 Q (then logits / P)
constexpr uint32_t kOffK = 0, kOffQ = kTileBytes, kOffMisc = kOffQ + kQBytes;
constexpr uint32_t kMiscBytes = 1792;
constexpr uint32_t kSmemBytes = kOffMisc + kMiscBytes + 1024;   // + alignment slack
constexpr size_t kPartFloats = (size_t)kHAtt * kDLat + 2 * kHAtt;   // one CTA's partial in the workspace
constexpr uint32_t kOffPinQ = 40960;                     // P inside the Q region (the softmax exchange sits below it)
constexpr int kTmemCols = 512;
constexpr int kColS = 0, kColO = 256;                    // S [64 heads][160 keys], O^T [4 x 128 dims][64 heads]
constexpr int kKeysPerWarp = kRows / 4;                  // softmax: the 4 warps of a TMEM lane quadrant split the keys
static_assert(kSmemBytes <= 232448, "shared memory");
static_assert(kOffPinQ % 1024 == 0 && 512 * 4 <= (int)kOffPinQ, "softmax exchange below P");
static_assert(kKeysPerWarp == 40 && kColS + kRows <= kColO, "S columns");
static_assert(kOffPinQ + 3 * kHAtt * 128 <= kQBytes, "P^T (160 keys in three 64-key blocks)");


// store a float pair to the same shared-memory variable in CTA `peer` of the cluster
__device__ __forceinline__ void st_cluster_f2(uint32_t local_addr, uint32_t peer, float a, float b) {
  asm volatile(
      "{ .reg .b32 ra; mapa.shared::cluster.u32 ra, %0, %1; st.shared::cluster.v2.f32 [ra], {%2, %3}; }" ::"r"(
          local_addr),
      "r"(peer), "f"(a), "f"(b)
      : "memory");
}
// elementwise max(m, |x|) on bf16 pairs
__device__ __forceinline__ uint32_t bf16x2_max_abs(uint32_t m, uint32_t x) {
  const __nv_bfloat162 r = __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&m),
                                   __habs2(*reinterpret_cast<const __nv_bfloat162*>(&x)));
  return *reinterpret_cast<const uint32_t*>(&r);
}
// 2-D tiled TMA load of one box into this CTA's shared memory; the mbarrier at `bar` receives
// the byte count
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
// cluster barrier arrive without release semantics: for a thread that published nothing, or
// that already ordered what it published with fence_cluster()
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void fence_cluster() { asm volatile("fence.acq_rel.cluster;" ::: "memory"); }
// Plain global loads (coherent, cached in L1) for the gathered cache rows, which the cache
// writer may have produced: unlike ld.global.nc they cannot be served before the dependency wait
// (the L2-only ld.global.cg costs 6 % of the decode step here)
__device__ __forceinline__ uint4 ld_global_v4(const uint4* ptr) {
  uint4 v;
  asm volatile("ld.global.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(ptr));
  return v;
}
__device__ __forceinline__ uint32_t ld_global_u16(const uint16_t* ptr) {
  unsigned short v;
  asm volatile("ld.global.u16 %0, [%1];" : "=h"(v) : "l"(ptr));
  return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t s2) {
  const __half2 r = __hmul2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&s2));
  return *reinterpret_cast<const uint32_t*>(&r);
}

__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kAttnThreads, 1)
    sparse_attn_kernel(const __grid_constant__ AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;      // 1024-byte alignment for the swizzled tiles
  uint8_t* sm = smem_raw + (base - raw_base);
  const uint32_t sK = base + kOffK, sQ = base + kOffQ, sP = base + kOffQ + kOffPinQ;
  float* misc = reinterpret_cast<float*>(sm + kOffMisc);
  float* s_scale = misc;              // [64] logit scale per head (read while staging the logits)
  float* s_invl = misc;               // [64] then 1 / l of this CTA's keys per head (read by the drain)
  float2* s_ml = reinterpret_cast<float2*>(misc + 64);   // [4 CTAs][16 own heads] (m_c, l_c), written by peers
  float* s_w = misc + 192;            // [4][16] combine weights of this CTA's heads
  int* s_valid = reinterpret_cast<int*>(misc + 256);      // [160]
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(misc + 416);
  // mbarriers: [0] QK done, [1..4] PV tile done, [5..8] K-tile step s converted (all 16 warps),
  // [9] query landed (64 KB)
  const uint32_t bar = smem_u32(misc + 418);
  const uint32_t kb_bar = bar + 8u * 5;
  const uint32_t q_bar = bar + 8u * 9;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_rank();
  const int row = blockIdx.x / kCluster;              // (b, q) flattened
  const int b = row / p.nq, qi = row % p.nq;
  // workspace partial of CTA c: [32 head pairs][512 dims] f16x2 (the pairs it does not own)
  uint32_t* part = reinterpret_cast<uint32_t*>(p.partial + ((size_t)row * kCluster) * kPartFloats);

  // ---------------------------------------------------------------- setup (overlaps the previous kernel)
  if (warp == 0) {
    tmem_alloc(smem_u32(s_tmem), kTmemCols);
  }
  if (tid == 0) {
#pragma unroll
    for (int i = 0; i < 5; ++i) mbar_init(bar + 8u * i, 1);
#pragma unroll
    for (int i = 0; i < 4; ++i) mbar_init(kb_bar + 8u * i, kWorkWarps);
    mbar_init(q_bar, 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // Peers store into this CTA's (m, l) slots only once it runs: the matching wait comes right
  // before each thread's first store into a peer (or, for the MMA warp, before phase A). The
  // arrive publishes nothing (the barriers are CTA-local), so it is relaxed.
  cluster_arrive_relaxed();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(s_tmem);
  // query: all 64 heads, 8 boxes of 64 dims x 64 heads (8 KB each), into this CTA's own shared
  // memory
  auto issue_query = [&]() {
    if (warp == kWorkWarps && lane == 0) {
      mbar_arrive_expect_tx(q_bar, kQBytes);
#pragma unroll
      for (int kb = 0; kb < 8; ++kb)
        tma_load_2d(sQ + (uint32_t)kb * (kHAtt * 128u), &p.qmap, 64 * kb, row * kHAtt, q_bar);
    }
  };
  // SWA: this CTA's 32 window rows (w = 32 rank + r, position vis - 128 + w) are one contiguous
  // 16 KB block; worker warp w takes rows 8 (w >> 2) + rr, FP8 chunks jj = 4 (2 (w & 3) + s) + qq
  // (lane = 8 qq + rr)
  const int rr = lane & 7, qq = lane >> 3;
  const int srow = 8 * (warp >> 2) + rr;
  uint4 sc[2];
  auto load_swa = [&]() {
    if (warp < kWorkWarps) {
      const uint4* src = reinterpret_cast<const uint4*>(
          p.swa + ((size_t)b * (kSwa + p.nq - 1) + qi + 32 * (int)rank + srow) * kDLat);
#pragma unroll
      for (int s4 = 0; s4 < 2; ++s4) sc[s4] = __ldg(src + 4 * (2 * (warp & 3) + s4) + qq);
    }
  };
  // Inputs that no kernel of the same step writes (schedule_step) are fetched while the previous
  // kernel drains; otherwise only after the programmatic-dependency wait. Nothing is written to
  // global memory before that wait.
  if (p.inputs_ready) {
    issue_query();
    load_swa();
  }
  // A Reuse slot of schedule_step reads nothing the previous kernel wrote (its top-k is two or
  // more kernels old): it waits only before its first global write, the partials drain.
  // The next kernel is released once the key tile is converted (worker warps) and QK is issued
  // (MMA warp), not here: released at the top, its early CTAs' loads compete with this kernel's
  // gathers while its later CTAs still wait for SMs (measured: 0.5 % slower per step; with no
  // release before exit, 6 % slower).
  if (!p.topk_ready) griddep_wait();
  if (!p.inputs_ready) {
    issue_query();
    load_swa();
  }

  if (warp == kWorkWarps) {
    // ---------------------------------------------------------------- MMA warp
    if (lane == 0) {
      // S = Q . K^T: M = 64 heads (A = the query, K-major), N = 160 keys (B = the tile, K-major),
      // 128-dim step by step as the worker warps finish converting them. Descriptors are formed
      // once; a k-step only moves the start-address field (address >> 4), which cannot carry out
      // of its 14 bits because every operand lies below 256 KB.
      const uint32_t id = idesc_f16(64, kRows, false, false);
      const uint64_t a0 = sdesc(sQ, 16u, 1024u), b0 = sdesc(sK, 16u, 1024u);
      bool ok = true;
#pragma unroll
      for (int st = 0; st < 4; ++st) {
        ok = mbar_wait(kb_bar + 8u * st, 0, p.wait_ns) && ok;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const int k = 8 * st + kk;
          const uint32_t ko = ((uint32_t)(k >> 2) * kKbStride + (uint32_t)(k & 3) * 32u) >> 4;
          const uint32_t qo = ((uint32_t)(k >> 2) * (kHAtt * 128u) + (uint32_t)(k & 3) * 32u) >> 4;
          umma_f16(tmem + kColS, a0 + qo, b0 + ko, id, k > 0);
        }
      }
      umma_commit(bar);
      if (!ok) flag_status(p.status, HSA_FLAG_TIMEOUT);
    }
    __syncwarp();
    griddep_launch_dependents();
    named_bar_sync(2, kAttnThreads);  // P^T written by the worker warps
    if (lane == 0) {
      tc_fence_after();
      // O^T = V^T . P^T one M-tile (128 dims) at a time, each with its own completion barrier,
      // so the workers drain finished tiles while the tensor core works on the next ones
      const uint32_t id = idesc_f16(128, 64, true, false);
      const uint64_t a0 = sdesc(sK, kKbStride, 1024u), b0 = sdesc(sP, 16u, 1024u);
#pragma unroll
      for (int mt = 0; mt < 4; ++mt) {
#pragma unroll
        for (int ks = 0; ks < kRows / 16; ++ks) {
          const uint32_t bo = ((uint32_t)(ks >> 2) * (kHAtt * 128u) + (uint32_t)(ks & 3) * 32u) >> 4;
          const uint32_t ao = ((uint32_t)(2 * mt) * kKbStride + (uint32_t)(16 * ks) * 128u) >> 4;
          umma_f16(tmem + kColO + 64 * mt, a0 + ao, b0 + bo, id, ks > 0);
        }
        umma_commit(bar + 8u * (1 + mt));
      }
    }
    __syncwarp();
    cluster_wait();                   // setup barrier (arrived at the top)
    cluster_arrive_relaxed();         // phase A: (m, l) published (this warp stored none)
    cluster_wait();
    cluster_arrive_relaxed();         // phase B: partials published (this warp stored none)
    cluster_wait();
    return;
  }

  // ---------------------------------------------------------------- worker warps (0..15)
  const int vis = __ldg(p.vis + row);

  // issue every global load up front. Lane = 8 q + rr. One warp-wide load covers 8 rows (rr) x
  // 64 contiguous bytes (4 lanes q x 16 B), so every sector fetched is used whole, and in the
  // shared-memory stores that follow, the 8 lanes of each store phase write 8 different rows.
  // top-k rows: warp w owns rows 8w + rr; step s takes code chunk j = 4 s + qq (dims 32j..32j+31).
  // The row index goes first: the row loads depend on it. The indices and the cache rows are
  // other kernels' outputs: coherent loads only (see griddep_wait)
  const int krow = 8 * warp + rr;
  const int kidx = __ldcg(p.topk + (size_t)row * kTopK + rank * kTopRows + krow);
  const bool sval = (vis - kSwa + 32 * (int)rank + srow) >= 0;
  uint4 kc[4];
  uint32_t ks2[4];
  {
    // the gather address depends on the index alone (clamped into the cache); whether the row
    // counts (index in [0, vis)) is applied when it is converted
    const size_t e = (size_t)b * p.cap + (size_t)min(max(kidx, 0), (int)imin64(p.cap, 0x7fffffff) - 1);
#pragma unroll
    for (int s4 = 0; s4 < 4; ++s4) {
      const int j = 4 * s4 + qq;
      kc[s4] = ld_global_v4(reinterpret_cast<const uint4*>(p.kv_q + e * 256) + j);
      ks2[s4] = ld_global_u16(reinterpret_cast<const uint16_t*>(p.kv_s + e * 32) + j);
    }
  }

  const bool kval = (kidx >= 0) && (kidx < vis) && (kidx < p.cap);
  if (kidx >= 0 && !kval && qq == 0) flag_status(p.status, HSA_FLAG_INDEX_RANGE);

  // ---------------------------------------------------------------- q: bf16 -> f16 in place, per-head shift
  // Warp w owns heads 4w .. 4w+3 whole: lane = 8 hq + c reads 16-byte chunk c of each of the 8
  // 64-dim blocks of head 4w + hq (one phase of 8 lanes reads one 128-byte row: no conflicts),
  // takes the head's |q| max over its 8 lanes and writes the f16 values back to the same place.
  {
    const int qh = 4 * warp + (lane >> 3), c = lane & 7;
    const uint32_t a0 = sQ + sw128((uint32_t)qh, (uint32_t)c);
    if (!mbar_wait(q_bar, 0, p.wait_ns) && lane == 0) flag_status(p.status, HSA_FLAG_TIMEOUT);
    uint4 qv[8];
#pragma unroll
    for (int kb = 0; kb < 8; ++kb) qv[kb] = lds128(a0 + (uint32_t)kb * (kHAtt * 128u));
    uint32_t m2 = 0u;                 // bf16x2 running max of |q|
#pragma unroll
    for (int kb = 0; kb < 8; ++kb) {
      m2 = bf16x2_max_abs(m2, qv[kb].x);
      m2 = bf16x2_max_abs(m2, qv[kb].y);
      m2 = bf16x2_max_abs(m2, qv[kb].z);
      m2 = bf16x2_max_abs(m2, qv[kb].w);
    }
    float amax = fmaxf(__uint_as_float(m2 << 16), __uint_as_float(m2 & 0xFFFF0000u));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
    int sh = 0;
    if (amax > 0.f) {
      int e;
      frexpf(amax, &e);
      sh = max(-126, min(127, 15 - e));     // amax * 2^sh in [2^14, 2^15)
    }
    const float mul = __uint_as_float((uint32_t)(127 + sh) << 23);   // exact power of two
    if (c == 0) s_scale[qh] = p.sm_scale * __uint_as_float((uint32_t)(127 - sh) << 23);
#pragma unroll
    for (int kb = 0; kb < 8; ++kb) {
      const uint32_t w[4] = {qv[kb].x, qv[kb].y, qv[kb].z, qv[kb].w};
      uint32_t o[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const __half2 h = __floats2half2_rn(__uint_as_float(w[j] << 16) * mul,
                                            __uint_as_float(w[j] & 0xFFFF0000u) * mul);
        o[j] = *reinterpret_cast<const uint32_t*>(&h);
      }
      sts128(a0 + (uint32_t)kb * (kHAtt * 128u), o[0], o[1], o[2], o[3]);
    }
  }

  // ---------------------------------------------------------------- K tile: SWA rows (E4M3 -> f16, exact)
#pragma unroll
  for (int s4 = 0; s4 < 2; ++s4) {
    const int jj = 4 * (2 * (warp & 3) + s4) + qq;       // dims 16 jj .. 16 jj + 15
    const uint32_t vw[4] = {sc[s4].x, sc[s4].y, sc[s4].z, sc[s4].w};
    uint32_t o[8];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      o[2 * u] = sval ? e4m3x2_to_f16x2((uint16_t)(vw[u] & 0xFFFFu)) : 0u;
      o[2 * u + 1] = sval ? e4m3x2_to_f16x2((uint16_t)(vw[u] >> 16)) : 0u;
    }
    const int r = kTopRows + srow;
    const uint32_t blk = sK + (uint32_t)(jj >> 2) * kKbStride;
    const int c0 = 2 * (jj & 3);
    sts128(blk + sw128(r, c0), o[0], o[1], o[2], o[3]);
    sts128(blk + sw128(r, c0 + 1), o[4], o[5], o[6], o[7]);
  }
  if ((warp & 3) == 0 && qq == 0) s_valid[kTopRows + srow] = sval ? 1 : 0;

  // ---------------------------------------------------------------- K tile: top-k rows (E2M1 x scale -> f16)
  // Step s converts dims 128 s .. 128 s + 127 (blocks 2s, 2s+1) of this warp's 8 rows; after it
  // the warp arrives on step s's barrier, and the MMA warp runs that step's QK k-steps.
#pragma unroll
  for (int s4 = 0; s4 < 4; ++s4) {
    const int j = 4 * s4 + qq;
    const uint32_t cw[4] = {kc[s4].x, kc[s4].y, kc[s4].z, kc[s4].w};
    uint32_t o[16];
#pragma unroll
    for (int w = 0; w < 4; ++w) e2m1x8_to_f16x2x4(cw[w], o[4 * w], o[4 * w + 1], o[4 * w + 2], o[4 * w + 3]);
#pragma unroll
    for (int gi = 0; gi < 2; ++gi) {
      const uint32_t sb = (ks2[s4] >> (8 * gi)) & 0xFFu;
      const float sf = (p.scale_fmt == HSA_SCALE_E8M0) ? e8m0_to_f32(sb) : e4m3_to_f32(sb);
      const uint32_t s2 = kval ? (uint32_t)__half_as_ushort(__float2half_rn(sf)) * 0x10001u : 0u;
#pragma unroll
      for (int u = 0; u < 8; ++u) o[8 * gi + u] = hmul2_u32(o[8 * gi + u], s2);
    }
    // dims 32j + 8w -> block kb = j / 2, 16-byte chunk 4 (j & 1) + w
    const uint32_t blk = sK + (uint32_t)(j >> 1) * kKbStride;
#pragma unroll
    for (int w = 0; w < 4; ++w)
      sts128(blk + sw128(krow, 4 * (j & 1) + w), o[4 * w], o[4 * w + 1], o[4 * w + 2], o[4 * w + 3]);
    fence_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(kb_bar + 8u * s4);
  }
  if (qq == 0) s_valid[krow] = kval ? 1 : 0;
  griddep_launch_dependents();

  if (!mbar_wait(bar, 0, p.wait_ns) && tid == 0) flag_status(p.status, HSA_FLAG_TIMEOUT);
  tc_fence_after();
  named_bar_sync(1, kWorkThreads);    // s_valid, s_scale visible

  // ---------------------------------------------------------------- softmax, one head per TMEM lane
  // S[h][key] lies in TMEM lane 32 (h / 16) + h % 16 (the M = 64 accumulator layout), column key.
  // Warp w reads lane quadrant sq = w & 3 (heads 16 sq .. 16 sq + 15 in its lanes 0..15) and the
  // 40 keys 40 sj .. 40 sj + 39, sj = w >> 2; lanes 16..31 hold no head and only take part in the
  // collective loads and the barriers. The four warps of a quadrant merge their (max, sum)
  // through shared memory (below P in the query region, which QK has consumed).
  const int sq = warp & 3, sj = warp >> 2;
  const bool hl = lane < 16;
  const int hh = 16 * sq + (lane & 15);
  float* s_red = reinterpret_cast<float*>(sm + kOffQ);   // [2][4 key quarters][64 heads]: max, then sum
  float x[kKeysPerWarp];
  {
    uint32_t r[kKeysPerWarp];
    const uint32_t ta = tmem + ((uint32_t)(32 * sq) << 16) + (uint32_t)(kColS + kKeysPerWarp * sj);
    TMEM_LD32(ta, r);
    TMEM_LD8(ta + 32u, (r + 32));
    tmem_wait_ld();
    tmem_regs_ready(r);
    const float scl = s_scale[hh];
#pragma unroll
    for (int i = 0; i < kKeysPerWarp; ++i)
      x[i] = s_valid[kKeysPerWarp * sj + i] ? __uint_as_float(r[i]) * scl : -INFINITY;
  }
  float mloc = -INFINITY;
#pragma unroll
  for (int i = 0; i < kKeysPerWarp; ++i) mloc = fmaxf(mloc, x[i]);
  if (hl) s_red[sj * kHAtt + hh] = mloc;
  named_bar_sync(1, kWorkThreads);
  mloc = fmaxf(fmaxf(s_red[hh], s_red[kHAtt + hh]), fmaxf(s_red[2 * kHAtt + hh], s_red[3 * kHAtt + hh]));
  // P (f16) into the B operand [keys/64][64 heads][128 B]: rows = heads, K = keys; one 8-key run
  // is one 16-byte unit.
  // p = 2^(x log2 e - m log2 e); a head with no valid key has m = -inf and every x = -inf, so
  // its offset is 0 and every p is 0. Values below 2^-126 flush to zero (f16 P rounds everything
  // below 2^-25 to zero anyway). Key pairs run as packed fp32 pairs.
  const float kLog2e = 1.4426950408889634f;
  const float ml2 = (mloc == -INFINITY) ? 0.f : mloc * kLog2e;
  const uint64_t l2e2 = f2_pack(kLog2e, kLog2e), nml2 = f2_pack(-ml2, -ml2);
  uint64_t ls2 = f2_pack(0.f, 0.f);
#pragma unroll
  for (int u = 0; u < kKeysPerWarp / 8; ++u) {
    uint32_t pk[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float z0, z1;
      f2_unpack(f2_fma(f2_pack(x[8 * u + 2 * e], x[8 * u + 2 * e + 1]), l2e2, nml2), z0, z1);
      const float p0 = ex2_ftz(z0), p1 = ex2_ftz(z1);
      ls2 = f2_add(ls2, f2_pack(p0, p1));
      const __half2 h = __floats2half2_rn(p0, p1);
      pk[e] = *reinterpret_cast<const uint32_t*>(&h);
    }
    const int key = kKeysPerWarp * sj + 8 * u;
    if (hl) sts128(sP + (uint32_t)(key >> 6) * (kHAtt * 128u) + sw128(hh, (key & 63) >> 3), pk[0], pk[1], pk[2], pk[3]);
  }
  float lsum;
  {
    float a, c;
    f2_unpack(ls2, a, c);
    lsum = a + c;
  }
  if (hl) s_red[(4 + sj) * kHAtt + hh] = lsum;
  named_bar_sync(1, kWorkThreads);
  lsum = (s_red[4 * kHAtt + hh] + s_red[5 * kHAtt + hh]) + (s_red[6 * kHAtt + hh] + s_red[7 * kHAtt + hh]);
  const bool hown = hl && sj == 0;    // one thread per head publishes its (m, l)
  if (hown) s_invl[hh] = (lsum > 0.f) ? 1.f / lsum : 0.f;
  fence_async_smem();
  named_bar_sync(2, kAttnThreads);    // P ready for the MMA warp; s_invl visible to every worker
  // (m_c, l_c) of head hh go to the CTA that owns it (slot [rank][hh % 16]); read after phase A.
  // Every peer has started (setup barrier).
  cluster_wait();
  if (hown) st_cluster_f2(smem_u32(s_ml + rank * 16 + (hh & 15)), (uint32_t)(hh >> 4), mloc, lsum);
  uint32_t* mine = part + (size_t)rank * kPartFloats;
  // phase A: only warps 0..3 stored into peers ((m, l) of their heads); they release it with a
  // cluster-scope fence, so every thread's arrive can be relaxed
  if (warp < 4) fence_cluster();
  cluster_arrive_relaxed();

  // ---------------------------------------------------------------- partial O / l -> L2
  // Warp (quadrant qd = w & 3, tile mt = w >> 2) owns output dimension d = 128 mt + 32 qd + lane
  // for all 64 heads: it sends the 48 heads other CTAs combine to the workspace (L2) as f16,
  // [h / 8][d] units of 8 heads, and keeps this CTA's own 16 heads in registers (fp32).
  if (p.topk_ready) griddep_wait();   // the previous kernel may still read the partials workspace
  const int qd = warp & 3, mtile = warp >> 2;
  const int dim = 128 * mtile + 32 * qd + lane;
  float own[16];
  {
    if (!mbar_wait(bar + 8u * (1 + mtile), 0, p.wait_ns) && lane == 0) flag_status(p.status, HSA_FLAG_TIMEOUT);
    tc_fence_after();
#pragma unroll
    for (int hc = 0; hc < 2; ++hc) {
      uint32_t r[32];
      TMEM_LD32(tmem + ((uint32_t)(32 * qd) << 16) + (uint32_t)(kColO + 64 * mtile + 32 * hc), r);
      tmem_wait_ld();
      tmem_regs_ready(r);
      uint32_t pk[16];
#pragma unroll
      for (int j = 0; j < 32; j += 2) {
        const int h = 32 * hc + j;
        const float2 il = *reinterpret_cast<const float2*>(s_invl + h);
        float o0, o1;
        f2_unpack(f2_mul(f2_pack(__uint_as_float(r[j]), __uint_as_float(r[j + 1])), f2_pack(il.x, il.y)), o0, o1);
        if ((h >> 4) == (int)rank) {
          own[h & 15] = o0;
          own[(h & 15) + 1] = o1;
        }
        const __half2 v = __floats2half2_rn(o0, o1);
        pk[j >> 1] = *reinterpret_cast<const uint32_t*>(&v);
      }
      // 8 heads (4 pairs) per 16-byte unit: group G = 4 hc + u covers heads 8G .. 8G + 7
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int G = 4 * hc + u;
        if ((G >> 1) != (int)rank)
          __stcg(reinterpret_cast<uint4*>(mine) + (size_t)G * kDLat + dim,
                 make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]));
      }
    }
  }
  tc_fence_before();
  cluster_wait();                     // phase A: every CTA's (m, l) is visible
  // combine weights of this CTA's heads: w_c = exp(m_c - M) l_c / sum_c' exp(m_c' - M) l_c'
  if (tid < 16) {
    float mc[kCluster], lc[kCluster];
#pragma unroll
    for (int c = 0; c < kCluster; ++c) {
      const float2 ml = s_ml[c * 16 + tid];
      mc[c] = ml.x;
      lc[c] = ml.y;
    }
    float M = -INFINITY;
#pragma unroll
    for (int c = 0; c < kCluster; ++c) M = fmaxf(M, mc[c]);
    float e[kCluster], L = 0.f;
#pragma unroll
    for (int c = 0; c < kCluster; ++c) {
      e[c] = (mc[c] == -INFINITY) ? 0.f : exp2f((mc[c] - M) * 1.4426950408889634f);
      L += e[c] * lc[c];
    }
    const float inv = (L > 0.f) ? 1.f / L : 0.f;
#pragma unroll
    for (int c = 0; c < kCluster; ++c) s_w[c * 16 + tid] = e[c] * lc[c] * inv;
  }
  cluster_arrive();                   // phase B: this CTA's partial is published
  cluster_wait();
  tc_fence_after();
  if (warp == 0) {
    // Nothing of this CTA may still be in flight when it frees its tensor memory and exits, even
    // if a wait above gave up: the last PV commit covers every MMA the CTA issued, q_bar the
    // query copy (both waits are bounded, and immediate when nothing timed out).
    if (!mbar_wait(bar + 8u * 4, 0, p.wait_ns) && lane == 0) flag_status(p.status, HSA_FLAG_TIMEOUT);
    if (!mbar_wait(q_bar, 0, p.wait_ns) && lane == 0) flag_status(p.status, HSA_FLAG_TIMEOUT);
    tc_fence_after();
    tmem_free(tmem, kTmemCols);
  }

  // ---------------------------------------------------------------- out[h][dim] = sum_c w_c[h] O_c[h][dim], c in rank order
  {
    uint64_t acc2[8];                 // head pairs (j, j + 1) of this CTA's 16
#pragma unroll
    for (int j = 0; j < 8; ++j) acc2[j] = f2_pack(0.f, 0.f);
    float v[16];
#pragma unroll
    for (uint32_t c = 0; c < kCluster; ++c) {
      if (c == rank) {
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = own[j];
      } else {
        // this CTA's heads 16 rank .. + 15 are groups 2 rank and 2 rank + 1 of peer c's partial
        const uint4* src = reinterpret_cast<const uint4*>(part + (size_t)c * kPartFloats) + (size_t)(2 * rank) * kDLat + dim;
#pragma unroll
        for (int g2 = 0; g2 < 2; ++g2) {
          const uint4 u4 = __ldcg(src + (size_t)g2 * kDLat);
          const uint32_t uu[4] = {u4.x, u4.y, u4.z, u4.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&uu[j]));
            v[8 * g2 + 2 * j] = f.x;
            v[8 * g2 + 2 * j + 1] = f.y;
          }
        }
      }
#pragma unroll
      for (int j = 0; j < 16; j += 2) {
        const float2 wc = *reinterpret_cast<const float2*>(s_w + c * 16 + j);
        acc2[j >> 1] = f2_fma(f2_pack(wc.x, wc.y), f2_pack(v[j], v[j + 1]), acc2[j >> 1]);
      }
    }
    float* out = p.out + ((size_t)row * kHAtt + 16 * rank) * kDLat + dim;
#pragma unroll
    for (int j = 0; j < 16; j += 2) {
      float a, c;
      f2_unpack(acc2[j >> 1], a, c);
      out[(size_t)j * kDLat] = a;
      out[(size_t)(j + 1) * kDLat] = c;
    }
  }
}

}  // namespace

namespace {
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// the driver's tensor-map encoder, looked up once through the runtime (no libcuda link)
EncodeTiledFn encode_tiled() {
  static const EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  return fn;
}
}  // namespace

cudaError_t launch_attention(const AttnParams& p, cudaStream_t s) {
  cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(sparse_attn_kernel), kSmemBytes);
  if (e != cudaSuccess) return e;
  const int rows = p.batch * p.nq;
  const EncodeTiledFn encode = encode_tiled();
  if (!encode) return cudaErrorNotSupported;
  AttnParams a = p;
  // q viewed as [rows * 64 heads][512 dims] bf16: a box is 64 dims (128 B, the swizzle span) x 64 heads
  const cuuint64_t dims[2] = {(cuuint64_t)kDLat, (cuuint64_t)rows * kHAtt};
  const cuuint64_t strides[1] = {(cuuint64_t)kDLat * 2};
  const cuuint32_t box[2] = {64, 64};
  const cuuint32_t estr[2] = {1, 1};
  if (encode(&a.qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(p.q), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  return launch_pdl(sparse_attn_kernel, dim3(rows * kCluster), dim3(kAttnThreads), kSmemBytes, s, a);
}

}  // namespace hsa
