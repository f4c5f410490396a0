// Sparse attention over the selected FP4 main-KV rows plus the FP8 SWA tail
// ([CED] Figure 4: Selected Main KV ⊕ SWA KV -> Core Attention; [890B] 注意力实际有多稀:
// 512 + 128 = 640 positions; [ARCH] §7: dequantise before attention, no FP4 matmul needed).
//
// One thread-block cluster of 4 CTAs per (request, query). CTA j owns 160 keys: top-k slots
// [128j, 128j+128) and SWA window rows [32j, 32j+32). Four CTAs per row fit a batch of 32
// requests in one wave of 128 SMs. Each CTA:
//  1. issues every global load at once: its 160 rows (gathered once and shared by all 64
//     heads) and the 64x512 bf16 query. It dequantises the rows to f16 (E2M1 x scale, or E4M3
//     for SWA) into a 128B-swizzled K-major shared tile. The query is converted to f16 after a
//     per-head power-of-two shift (exact within f16), in the same layout;
//  2. tcgen05: S^T = K . Q^T in two M=128 passes (rows 0..127, then rows 32..159, of which only
//     keys 128..159 are used), accumulated in TMEM;
//  3. exchanges per-head max and sum through distributed shared memory, so every CTA
//     normalises against the global max. It writes P^T (f16) as the next B operand;
//  4. tcgen05: O^T[512 dims][64 heads] = V^T . P^T, reading the same tile as an MN-major
//     A operand (K = V = the 512-d latent), 4 M-tiles of 128 dims x 10 k-steps;
//  5. scales by 1/sum, stages its partial in shared memory, and sums its 16-head slice over
//     the 4 CTAs through DSMEM in a fixed order (deterministic).
// Setup (TMEM allocation, barrier init) runs before the programmatic-dependency wait, so it
// overlaps the tail of the previous kernel in the stream. Every wait is bounded.
#include "hsa_common.cuh"
#include "hsa_internal.h"

namespace hsa {
namespace {

constexpr int kAttnThreads = 256;
constexpr int kCluster = 4;
constexpr int kRows = 160;                               // keys per CTA
constexpr int kTopRows = 128;
constexpr uint32_t kKbStride = kRows * 128u;             // bytes per 64-dim block of the tile
constexpr uint32_t kTileBytes = 8 * kKbStride;           // 160 KB f16 tile
constexpr uint32_t kQBytes = kHAtt * kDLat * 2;          // 64 KB f16 Q (then logits / P)
constexpr uint32_t kOffK = 0, kOffQ = kTileBytes, kOffMisc = kOffQ + kQBytes;
constexpr uint32_t kMiscBytes = 1792;
constexpr uint32_t kSmemBytes = kOffMisc + kMiscBytes + 1024;   // + alignment slack
constexpr int kSStride = 164;                            // fp32 staging row stride (conflict-free)
constexpr int kTmemCols = 512;
constexpr int kColS0 = 0, kColS1 = 64, kColO = 256;
static_assert(kSmemBytes <= 232448, "shared memory");
static_assert(kHAtt * kSStride * 4 <= (int)kQBytes, "logit staging");

// ------------------------------------------------------------------ tcgen05 helpers
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  // tcgen05 shared-memory matrix descriptor, 128-byte swizzle
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}
// kind::f16 instruction descriptor: f16 x f16 -> f32, dense
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, bool acc) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0;\n"
      "  tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc ? 1u : 0u));
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

#define TMEM_LD32(taddr, r)                                                                                     \
  asm volatile(                                                                                                 \
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"          \
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"                                \
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),        \
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),  \
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),             \
        "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),             \
        "=r"(r[30]), "=r"(r[31])                                                                                \
      : "r"(taddr))
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t mapa(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ float ld_dsmem_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ float4 ld_dsmem_f32x4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ void sts16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}
// byte offset of the 16-byte chunk `chunk` (0..7) of row `row` inside a 128B-swizzled block
__device__ __forceinline__ uint32_t sw128(uint32_t row, uint32_t chunk) {
  return row * 128u + (((chunk ^ (row & 7u)) & 7u) << 4);
}
__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t s2) {
  const __half2 r = __hmul2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&s2));
  return *reinterpret_cast<const uint32_t*>(&r);
}

// 32 FP4 codes (two uint4) x four scale bytes -> 32 f16x2 (element 2j in the low half)
__device__ __forceinline__ void dequant_fp4_64(const uint4 c0, const uint4 c1, uint32_t sc4, int fmt, uint32_t* o) {
  const uint32_t cw[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
  for (int j = 0; j < 8; ++j) e2m1x8_to_f16x2x4(cw[j], o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
#pragma unroll
  for (int gi = 0; gi < 4; ++gi) {
    const uint32_t sb = (sc4 >> (8 * gi)) & 0xFFu;
    const float sf = (fmt == HSA_SCALE_E8M0) ? e8m0_to_f32(sb) : e4m3_to_f32(sb);
    const uint32_t s2 = (uint32_t)__half_as_ushort(__float2half_rn(sf)) * 0x10001u;
#pragma unroll
    for (int j = 0; j < 8; ++j) o[8 * gi + j] = hmul2_u32(o[8 * gi + j], s2);
  }
}

__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kAttnThreads, 1)
    sparse_attn_kernel(const AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;      // 1024-byte alignment for the swizzled tiles
  uint8_t* sm = smem_raw + (base - raw_base);
  const uint32_t sK = base + kOffK, sQ = base + kOffQ, sP = base + kOffQ;
  float* misc = reinterpret_cast<float*>(sm + kOffMisc);
  float* s_scale = misc;              // [64] logit scale per head
  float* s_m = misc + 64;             // [64] local max (read remotely)
  float* s_l = misc + 128;            // [64] local sum (read remotely)
  float* s_invl = misc + 192;         // [64]
  int* s_valid = reinterpret_cast<int*>(misc + 256);      // [160]
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(misc + 416);
  uint64_t* s_bar = reinterpret_cast<uint64_t*>(misc + 418);
  const uint32_t bar = smem_u32(s_bar);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_rank();
  const int row = blockIdx.x / kCluster;              // (b, q) flattened
  const int b = row / p.nq, qi = row % p.nq;

  // ---------------------------------------------------------------- setup (overlaps the previous kernel)
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(s_tmem)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  griddep_wait();
  griddep_launch_dependents();
  const int vis = __ldg(p.vis + row);

  // ---------------------------------------------------------------- issue every global load up front
  // warp = 64-dim segment kb; top-k rows r = lane + 32 i (i < 4), SWA row 128 + lane
  const int kb = warp;
  uint4 kr[4][2];
  uint32_t ksc[4];
  bool kval[4];
  {
    int idx[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) idx[i] = __ldg(p.topk + (size_t)row * kTopK + rank * kTopRows + lane + 32 * i);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      kval[i] = (idx[i] >= 0) && (idx[i] < vis) && (idx[i] < p.cap);
      if (idx[i] >= 0 && !kval[i] && kb == 0) flag_status(p.status, HSA_FLAG_INDEX_RANGE);
      const size_t e = (size_t)b * p.cap + (kval[i] ? idx[i] : 0);
      const uint4* cs = reinterpret_cast<const uint4*>(p.kv_q + e * 256 + kb * 32);
      kr[i][0] = __ldg(cs);
      kr[i][1] = __ldg(cs + 1);
      ksc[i] = __ldg(reinterpret_cast<const uint32_t*>(p.kv_s + e * 32 + kb * 4));
    }
  }
  // SWA: window row w = 32 rank + lane of this query holds position vis - 128 + w
  const int wrow = 32 * (int)rank + lane;
  const bool sval = (vis - kSwa + wrow) >= 0;
  uint4 sr[4];
  {
    const uint4* cs = reinterpret_cast<const uint4*>(
        p.swa + ((size_t)b * (kSwa + p.nq - 1) + qi + wrow) * kDLat + kb * 64);
#pragma unroll
    for (int j = 0; j < 4; ++j) sr[j] = __ldg(cs + j);
  }
  const int qh = tid >> 2, qk = tid & 3;    // Q: 4 threads per head, 128 dims each
  uint4 qraw[16];
  {
    const uint4* src = reinterpret_cast<const uint4*>(p.q + ((size_t)row * kHAtt + qh) * kDLat + qk * 128);
#pragma unroll
    for (int i = 0; i < 16; ++i) qraw[i] = __ldg(src + i);
  }

  // ---------------------------------------------------------------- K tile rows
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = lane + 32 * i;
    uint32_t o[32];
    dequant_fp4_64(kr[i][0], kr[i][1], ksc[i], p.scale_fmt, o);
    if (!kval[i]) {
#pragma unroll
      for (int j = 0; j < 32; ++j) o[j] = 0u;
    }
    if (kb == 0) s_valid[r] = kval[i] ? 1 : 0;
    const uint32_t blk = sK + (uint32_t)kb * kKbStride;
#pragma unroll
    for (int c = 0; c < 8; ++c) sts128(blk + sw128(r, c), o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
  }
  {
    const int r = kTopRows + lane;
    uint32_t o[32];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t vw[4] = {sr[j].x, sr[j].y, sr[j].z, sr[j].w};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        o[8 * j + 2 * u] = sval ? e4m3x2_to_f16x2((uint16_t)(vw[u] & 0xFFFFu)) : 0u;
        o[8 * j + 2 * u + 1] = sval ? e4m3x2_to_f16x2((uint16_t)(vw[u] >> 16)) : 0u;
      }
    }
    if (kb == 0) s_valid[r] = sval ? 1 : 0;
    const uint32_t blk = sK + (uint32_t)kb * kKbStride;
#pragma unroll
    for (int c = 0; c < 8; ++c) sts128(blk + sw128(r, c), o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
  }

  // ---------------------------------------------------------------- Q: bf16 -> f16 with per-head shift
  {
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint32_t w[4] = {qraw[i].x, qraw[i].y, qraw[i].z, qraw[i].w};
#pragma unroll
      for (int j = 0; j < 4; ++j)
        amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(w[j] << 16)), fabsf(__uint_as_float(w[j] & 0xFFFF0000u))));
    }
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    int sh = 0;
    if (amax > 0.f) {
      int e;
      frexpf(amax, &e);
      sh = max(-126, min(127, 15 - e));     // amax * 2^sh in [2^14, 2^15)
    }
    const float mul = __uint_as_float((uint32_t)(127 + sh) << 23);   // exact power of two
    if (qk == 0) s_scale[qh] = p.sm_scale * __uint_as_float((uint32_t)(127 - sh) << 23);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint32_t w[4] = {qraw[i].x, qraw[i].y, qraw[i].z, qraw[i].w};
      uint32_t o[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const __half lo = __float2half_rn(__uint_as_float(w[j] << 16) * mul);
        const __half hi = __float2half_rn(__uint_as_float(w[j] & 0xFFFF0000u) * mul);
        o[j] = (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
      }
      const int d = qk * 128 + i * 8;
      sts128(sQ + (uint32_t)(d >> 6) * (kHAtt * 128u) + sw128(qh, (d & 63) >> 3), o[0], o[1], o[2], o[3]);
    }
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(s_tmem);

  // ---------------------------------------------------------------- S^T = K . Q^T (two M=128 passes)
  if (tid == 0) {
    const uint32_t id = idesc_f16(128, 64, false, false);
#pragma unroll 1
    for (int pass = 0; pass < 2; ++pass) {
      const uint32_t row0 = pass ? 32u : 0u;
#pragma unroll 1
      for (int k = 0; k < kDLat / 16; ++k) {
        const uint32_t kbk = k >> 2, kk = k & 3;
        const uint64_t a = sdesc(sK + kbk * kKbStride + row0 * 128u + kk * 32u, 16u, 1024u);
        const uint64_t bq = sdesc(sQ + kbk * (kHAtt * 128u) + kk * 32u, 16u, 1024u);
        umma_f16(tmem + (pass ? kColS1 : kColS0), a, bq, id, k > 0);
      }
    }
    umma_commit(bar);
  }
  if (!mbar_wait(bar, 0) && tid == 0) flag_status(p.status, HSA_FLAG_TIMEOUT);
  tc_fence_after();

  // ---------------------------------------------------------------- logits -> staging [h][key] (Q region)
  float* stg = reinterpret_cast<float*>(sm + kOffQ);
  if (warp < 4 || warp == 7) {
    // warps 0..3: keys 32w + lane from pass 0; warp 7: keys 128 + lane = pass-1 rows 96 + lane
    const int qd = warp & 3;
    const int key = (warp < 4) ? 32 * qd + lane : kTopRows + lane;
    const uint32_t col = (warp < 4) ? kColS0 : kColS1;
    const bool kv = s_valid[key] != 0;
#pragma unroll
    for (int hc = 0; hc < 2; ++hc) {
      uint32_t r[32];
      TMEM_LD32(tmem + ((uint32_t)(32 * qd) << 16) + col + 32u * hc, r);
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int h = 32 * hc + j;
        stg[h * kSStride + key] = kv ? __uint_as_float(r[j]) * s_scale[h] : -INFINITY;
      }
    }
  }
  __syncthreads();
  // per head: 4 threads, keys 4i + kq
  const int hh = tid >> 2, kq = tid & 3;
  float x[kRows / 4];
  float mloc = -INFINITY;
#pragma unroll
  for (int i = 0; i < kRows / 4; ++i) {
    x[i] = stg[hh * kSStride + 4 * i + kq];
    mloc = fmaxf(mloc, x[i]);
  }
  mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, 1));
  mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, 2));
  if (kq == 0) s_m[hh] = mloc;
  cluster_sync();               // publishes s_m; every thread has read its logits
  float M = -INFINITY;
#pragma unroll
  for (uint32_t src = 0; src < kCluster; ++src) M = fmaxf(M, ld_dsmem_f32(mapa(smem_u32(s_m + hh), src)));
  float lsum = 0.f;
  // P^T (f16) into the B operand [keys/64][64 heads][128 B]: rows = heads, K = keys
#pragma unroll
  for (int i = 0; i < kRows / 4; ++i) {
    const int key = 4 * i + kq;
    const float pr = (M == -INFINITY) ? 0.f : exp2f((x[i] - M) * 1.4426950408889634f);
    const __half ph = __float2half_rn(pr);
    lsum += __half2float(ph);                   // the value the tensor core will see
    sts16(sP + (uint32_t)(key >> 6) * (kHAtt * 128u) + sw128(hh, (key & 63) >> 3) + (uint32_t)(key & 7) * 2u,
          __half_as_ushort(ph));
  }
  lsum += __shfl_xor_sync(0xffffffffu, lsum, 1);
  lsum += __shfl_xor_sync(0xffffffffu, lsum, 2);
  if (kq == 0) s_l[hh] = lsum;
  fence_async_smem();
  tc_fence_before();
  cluster_sync();               // publishes s_l; P complete
  tc_fence_after();
  if (kq == 0) {
    float L = 0.f;
#pragma unroll
    for (uint32_t src = 0; src < kCluster; ++src) L += ld_dsmem_f32(mapa(smem_u32(s_l + hh), src));
    s_invl[hh] = (L > 0.f) ? 1.f / L : 0.f;
  }

  // ---------------------------------------------------------------- O^T = V^T . P^T
  if (tid == 0) {
    const uint32_t id = idesc_f16(128, 64, true, false);
#pragma unroll 1
    for (int mt = 0; mt < 4; ++mt) {
#pragma unroll 1
      for (int ks = 0; ks < kRows / 16; ++ks) {
        const uint64_t a = sdesc(sK + (uint32_t)(2 * mt) * kKbStride + (uint32_t)(16 * ks) * 128u, kKbStride, 1024u);
        const uint64_t bp = sdesc(sP + (uint32_t)(ks >> 2) * (kHAtt * 128u) + (uint32_t)(ks & 3) * 32u, 16u, 1024u);
        umma_f16(tmem + kColO + 64 * mt, a, bp, id, ks > 0);
      }
    }
    umma_commit(bar);
  }
  if (!mbar_wait(bar, 1) && tid == 0) flag_status(p.status, HSA_FLAG_TIMEOUT);
  tc_fence_after();
  __syncthreads();              // s_invl visible

  // ---------------------------------------------------------------- partial O (scaled) -> staging F[h][d] (K region)
  float* F = reinterpret_cast<float*>(sm + kOffK);
  {
    const int qd = warp & 3, half = warp >> 2;
#pragma unroll 1
    for (int u = 0; u < 2; ++u) {
      const int mt = 2 * half + u;
      const int d = 128 * mt + 32 * qd + lane;
#pragma unroll
      for (int hc = 0; hc < 2; ++hc) {
        uint32_t r[32];
        TMEM_LD32(tmem + ((uint32_t)(32 * qd) << 16) + (uint32_t)(kColO + 64 * mt + 32 * hc), r);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int h = 32 * hc + j;
          F[h * kDLat + d] = __uint_as_float(r[j]) * s_invl[h];
        }
      }
    }
  }
  tc_fence_before();
  cluster_sync();

  // ---------------------------------------------------------------- sum the cluster's partials for this CTA's 16 heads
  {
    float* out = p.out + (size_t)row * kHAtt * kDLat;
    const uint32_t Fs = smem_u32(F);
    constexpr int kPer = 16 * (kDLat / 4) / kAttnThreads;   // 8 float4 per thread
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      float4 v[kCluster][kPer / 2];
#pragma unroll
      for (int u = 0; u < kPer / 2; ++u) {
        const int i = tid + kAttnThreads * (hf * (kPer / 2) + u);
        const int h = 16 * (int)rank + i / (kDLat / 4), d4 = i % (kDLat / 4);
        const uint32_t off = Fs + (uint32_t)(h * kDLat + 4 * d4) * 4u;
#pragma unroll
        for (uint32_t src = 0; src < kCluster; ++src) v[src][u] = ld_dsmem_f32x4(mapa(off, src));
      }
#pragma unroll
      for (int u = 0; u < kPer / 2; ++u) {
        float4 acc = v[0][u];
#pragma unroll
        for (int src = 1; src < kCluster; ++src) {
          acc.x += v[src][u].x;
          acc.y += v[src][u].y;
          acc.z += v[src][u].z;
          acc.w += v[src][u].w;
        }
        const int i = tid + kAttnThreads * (hf * (kPer / 2) + u);
        const int h = 16 * (int)rank + i / (kDLat / 4), d4 = i % (kDLat / 4);
        reinterpret_cast<float4*>(out + (size_t)h * kDLat)[d4] = acc;
      }
    }
  }
  cluster_sync();
  tc_fence_after();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
}

}  // namespace

cudaError_t launch_attention(const AttnParams& p, cudaStream_t s) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(sparse_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int rows = p.batch * p.nq;
  return launch_pdl(sparse_attn_kernel, dim3(rows * kCluster), dim3(kAttnThreads), kSmemBytes, s, p);
}

}  // namespace hsa
