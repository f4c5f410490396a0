// Sparse attention over the selected FP4 main-KV rows plus the FP8 SWA tail
// ([CED] Figure 4: Selected Main KV ⊕ SWA KV -> Core Attention; [890B] 注意力实际有多稀:
// 512 + 128 = 640 positions; [ARCH] §7: dequantise before attention, no FP4 matmul needed).
//
// One thread-block cluster of 5 CTAs per (request, query); CTA j < 4 owns top-k slots
// [128j, 128j+128) and CTA 4 owns the 128 SWA rows. Each CTA:
//  1. gathers its 128 rows once and dequantises them to f16 (E2M1 x scale, or E4M3 for SWA)
//     into a 128B-swizzled K-major shared tile. The rows are shared by all 64 heads;
//  2. converts the 64x512 bf16 query to f16 after a per-head power-of-two shift (exact
//     within f16), in the same layout;
//  3. tcgen05: S^T[128 keys][64 heads] = K . Q^T (M=128, N=64, K=512), accumulated in TMEM;
//  4. exchanges per-head max and sum through distributed shared memory, so every CTA turns
//     its logits into probabilities against the global max. It writes P^T (f16) as the next
//     B operand;
//  5. tcgen05: O^T[512 dims][64 heads] = V^T . P^T, reading the same shared tile as an
//     MN-major A operand (K = V = the 512-d latent), 4 M-tiles of 128 dims in TMEM;
//  6. scales by 1/sum, stages its partial in shared memory and sums its 13-head slice of
//     the output over the 5 CTAs through DSMEM in a fixed order (deterministic).
// Every wait is bounded; a timeout sets HSA_FLAG_TIMEOUT and the CTA carries on to the end.
#include "hsa_common.cuh"
#include "hsa_internal.h"

namespace hsa {
namespace {

constexpr int kAttnThreads = 256;
constexpr int kCluster = 5;
constexpr int kKeys = 128;
constexpr uint32_t kTileBytes = kKeys * kDLat * 2;       // 128 KB f16 K tile
constexpr uint32_t kQBytes = kHAtt * kDLat * 2;          // 64 KB f16 Q
constexpr uint32_t kPBytes = kHAtt * kKeys * 2;          // 16 KB f16 P
constexpr uint32_t kOffK = 0, kOffQ = kTileBytes, kOffP = kOffQ + kQBytes, kOffMisc = kOffP + kPBytes;
constexpr uint32_t kSmemBytes = kOffMisc + 2048 + 1024;  // + 1 KB alignment slack
constexpr int kSStride = 132;                            // fp32 staging row stride (conflict-free)
constexpr int kTmemCols = 512;
constexpr int kColO = 256;

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
// byte offset of the 16-byte chunk `chunk` (0..7) of row `row` inside a 128B-swizzled block
__device__ __forceinline__ uint32_t sw128(uint32_t row, uint32_t chunk) {
  return row * 128u + (((chunk ^ (row & 7u)) & 7u) << 4);
}
__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t s2) {
  const __half2 r = __hmul2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&s2));
  return *reinterpret_cast<const uint32_t*>(&r);
}

__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kAttnThreads, 1)
    sparse_attn_kernel(const AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment for the swizzled operand tiles
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sm = smem_raw + (base - raw);
  const uint32_t sK = base + kOffK, sQ = base + kOffQ, sP = base + kOffP;
  float* misc = reinterpret_cast<float*>(sm + kOffMisc);
  float* s_scale = misc;              // [64] logit scale per head
  float* s_m = misc + 64;             // [64] local max (read remotely)
  float* s_l = misc + 128;            // [64] local sum (read remotely)
  float* s_invl = misc + 192;         // [64]
  int* s_valid = reinterpret_cast<int*>(misc + 256);   // [128]
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(misc + 384);
  uint64_t* s_bar = reinterpret_cast<uint64_t*>(misc + 388);   // 8-byte aligned
  const uint32_t bar = smem_u32(s_bar);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_rank();
  const int row = blockIdx.x / kCluster;            // (b, q) flattened
  const int b = row / p.nq, qi = row % p.nq;
  const int vis = __ldg(p.vis + row);

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(s_tmem)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }

  // ---------------------------------------------------------------- issue every global load up front
  // K rows: warp = 64-dim segment kb, 4 keys per thread (r = lane + 32 i)
  const int kb = warp;
  uint4 krow[4][4];
  uint32_t rsc[4];
  bool valid[4];
  if (rank < 4) {
    int idx[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) idx[i] = __ldg(p.topk + (size_t)row * kTopK + rank * kKeys + lane + 32 * i);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      valid[i] = (idx[i] >= 0) && (idx[i] < vis) && (idx[i] < p.cap);
      if (idx[i] >= 0 && !valid[i] && kb == 0) flag_status(p.status, HSA_FLAG_INDEX_RANGE);
      const size_t e = (size_t)b * p.cap + (valid[i] ? idx[i] : 0);
      const uint4* cs = reinterpret_cast<const uint4*>(p.kv_q + e * 256 + kb * 32);
      krow[i][0] = __ldg(cs);
      krow[i][1] = __ldg(cs + 1);
      rsc[i] = __ldg(reinterpret_cast<const uint32_t*>(p.kv_s + e * 32 + kb * 4));
    }
  } else {
    // SWA row r holds position vis - 128 + r for this query (rows [qi, qi+128) of the buffer)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = lane + 32 * i;
      valid[i] = (vis - kSwa + r) >= 0;
      const uint4* cs = reinterpret_cast<const uint4*>(
          p.swa + ((size_t)b * (kSwa + p.nq - 1) + qi + r) * kDLat + kb * 64);
#pragma unroll
      for (int j = 0; j < 4; ++j) krow[i][j] = __ldg(cs + j);
    }
  }
  // Q: 4 threads per head, 128 dims each
  const int qh = tid >> 2, qk = tid & 3;
  uint4 qraw[16];
  {
    const uint4* src = reinterpret_cast<const uint4*>(p.q + ((size_t)row * kHAtt + qh) * kDLat + qk * 128);
#pragma unroll
    for (int i = 0; i < 16; ++i) qraw[i] = __ldg(src + i);
  }

  // ---------------------------------------------------------------- Q: bf16 -> f16 with per-head shift
  {
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint32_t w[4] = {qraw[i].x, qraw[i].y, qraw[i].z, qraw[i].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(w[j] << 16)),
                                                           fabsf(__uint_as_float(w[j] & 0xFFFF0000u))));
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
      const int d = qk * 128 + i * 8;            // first dim of this 8-dim chunk
      const uint32_t addr = sQ + (uint32_t)(d >> 6) * (kHAtt * 128u) + sw128(qh, (d & 63) >> 3);
      sts128(addr, o[0], o[1], o[2], o[3]);
    }
  }

  // ---------------------------------------------------------------- K tile: dequantise into the swizzled tile
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = lane + 32 * i;
    uint32_t o[32];
    if (rank < 4) {
      const uint32_t cw[8] = {krow[i][0].x, krow[i][0].y, krow[i][0].z, krow[i][0].w,
                              krow[i][1].x, krow[i][1].y, krow[i][1].z, krow[i][1].w};
#pragma unroll
      for (int j = 0; j < 8; ++j) e2m1x8_to_f16x2x4(cw[j], o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
#pragma unroll
      for (int gi = 0; gi < 4; ++gi) {
        const uint32_t sb = (rsc[i] >> (8 * gi)) & 0xFFu;
        const float sf = (p.scale_fmt == HSA_SCALE_E8M0) ? e8m0_to_f32(sb) : e4m3_to_f32(sb);
        const __half hs = __float2half_rn(sf);
        const uint32_t s2 = (uint32_t)__half_as_ushort(hs) * 0x10001u;
#pragma unroll
        for (int j = 0; j < 8; ++j) o[8 * gi + j] = hmul2_u32(o[8 * gi + j], s2);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t vw[4] = {krow[i][j].x, krow[i][j].y, krow[i][j].z, krow[i][j].w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          o[8 * j + 2 * u] = e4m3x2_to_f16x2((uint16_t)(vw[u] & 0xFFFFu));
          o[8 * j + 2 * u + 1] = e4m3x2_to_f16x2((uint16_t)(vw[u] >> 16));
        }
      }
    }
    if (!valid[i]) {
#pragma unroll
      for (int j = 0; j < 32; ++j) o[j] = 0u;
    }
    if (kb == 0) s_valid[r] = valid[i] ? 1 : 0;
    const uint32_t blk = sK + (uint32_t)kb * (kKeys * 128u);
#pragma unroll
    for (int c = 0; c < 8; ++c) sts128(blk + sw128(r, c), o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(s_tmem);

  // ---------------------------------------------------------------- S^T = K . Q^T
  if (tid == 0) {
    const uint32_t id = idesc_f16(128, 64, false, false);
#pragma unroll 1
    for (int k = 0; k < kDLat / 16; ++k) {
      const uint32_t kb = k >> 2, kk = k & 3;
      const uint64_t a = sdesc(sK + kb * (kKeys * 128u) + kk * 32u, 16u, 1024u);
      const uint64_t bq = sdesc(sQ + kb * (kHAtt * 128u) + kk * 32u, 16u, 1024u);
      umma_f16(tmem, a, bq, id, k > 0);
    }
    umma_commit(bar);
  }
  bool ok = mbar_wait(bar, 0);
  if (!ok && tid == 0) flag_status(p.status, HSA_FLAG_TIMEOUT);
  tc_fence_after();

  // ---------------------------------------------------------------- logits -> staging [h][key] (Q region)
  float* stg = reinterpret_cast<float*>(sm + kOffQ);
  {
    const int qd = warp & 3, ch = warp >> 2;
    uint32_t r[32];
    TMEM_LD32(tmem + ((uint32_t)(32 * qd) << 16) + (uint32_t)(32 * ch), r);
    tmem_wait_ld();
    const int key = 32 * qd + lane;
    const bool kv = s_valid[key] != 0;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const int h = 32 * ch + j;
      stg[h * kSStride + key] = kv ? __uint_as_float(r[j]) * s_scale[h] : -INFINITY;
    }
  }
  __syncthreads();
  // per head: 4 threads, keys 4i + k
  const int hh = tid >> 2, kq = tid & 3;
  float mloc = -INFINITY;
  for (int i = 0; i < 32; ++i) mloc = fmaxf(mloc, stg[hh * kSStride + 4 * i + kq]);
  mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, 1));
  mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, 2));
  if (kq == 0) s_m[hh] = mloc;
  cluster_sync();
  float M = -INFINITY;
  for (uint32_t src = 0; src < kCluster; ++src) M = fmaxf(M, ld_dsmem_f32(mapa(smem_u32(s_m + hh), src)));
  float lsum = 0.f;
  for (int i = 0; i < 32; ++i) {
    const int key = 4 * i + kq;
    const float x = stg[hh * kSStride + key];
    float pr = (M == -INFINITY) ? 0.f : exp2f((x - M) * 1.4426950408889634f);
    pr = __half2float(__float2half_rn(pr));     // the value the tensor core will see
    lsum += pr;
    stg[hh * kSStride + key] = pr;
  }
  lsum += __shfl_xor_sync(0xffffffffu, lsum, 1);
  lsum += __shfl_xor_sync(0xffffffffu, lsum, 2);
  if (kq == 0) s_l[hh] = lsum;
  __syncthreads();
  // P^T (f16) into the B operand: rows = heads, K = keys; thread -> (head, 32-key quarter)
  {
    const int kq4 = tid & 3;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int k0 = 32 * kq4 + 8 * c;
      uint32_t o[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const __half lo = __float2half_rn(stg[hh * kSStride + k0 + 2 * u]);
        const __half hi = __float2half_rn(stg[hh * kSStride + k0 + 2 * u + 1]);
        o[u] = (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
      }
      const uint32_t addr = sP + (uint32_t)(k0 >> 6) * (kHAtt * 128u) + sw128(hh, (k0 & 63) >> 3);
      sts128(addr, o[0], o[1], o[2], o[3]);
    }
  }
  fence_async_smem();
  tc_fence_before();
  cluster_sync();               // also publishes s_l to the cluster
  tc_fence_after();
  if (kq == 0) {
    float L = 0.f;
    for (uint32_t src = 0; src < kCluster; ++src) L += ld_dsmem_f32(mapa(smem_u32(s_l + hh), src));
    s_invl[hh] = (L > 0.f) ? 1.f / L : 0.f;
  }

  // ---------------------------------------------------------------- O^T = V^T . P^T
  if (tid == 0) {
    const uint32_t id = idesc_f16(128, 64, true, false);
#pragma unroll 1
    for (int mt = 0; mt < 4; ++mt) {
#pragma unroll 1
      for (int kk = 0; kk < kKeys / 16; ++kk) {
        const uint64_t a = sdesc(sK + (uint32_t)(2 * mt) * (kKeys * 128u) + (uint32_t)(16 * kk) * 128u,
                                 kKeys * 128u, 1024u);
        const uint64_t bp = sdesc(sP + (uint32_t)(kk >> 2) * (kHAtt * 128u) + (uint32_t)(kk & 3) * 32u, 16u, 1024u);
        umma_f16(tmem + kColO + 64 * mt, a, bp, id, kk > 0);
      }
    }
    umma_commit(bar);
  }
  ok = mbar_wait(bar, 1);
  if (!ok && tid == 0) flag_status(p.status, HSA_FLAG_TIMEOUT);
  tc_fence_after();
  __syncthreads();              // s_invl visible

  // ---------------------------------------------------------------- partial O (scaled) -> staging F[h][d] (K region)
  float* F = reinterpret_cast<float*>(sm + kOffK);
  {
    const int qd = warp & 3, half = warp >> 2;
    for (int u = 0; u < 2; ++u) {
      const int mt = 2 * half + u;
      const int d = 128 * mt + 32 * qd + lane;
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

  // ---------------------------------------------------------------- sum the cluster's partials for this CTA's heads
  {
    const int hs = 13 * (int)rank, he = min(kHAtt, hs + 13);
    const int n4 = (he - hs) * (kDLat / 4);
    float* out = p.out + (size_t)row * kHAtt * kDLat;
    const uint32_t Fs = smem_u32(F);
    for (int i = tid; i < n4; i += kAttnThreads) {
      const int h = hs + i / (kDLat / 4), d4 = i % (kDLat / 4);
      const uint32_t off = Fs + (uint32_t)(h * kDLat + 4 * d4) * 4u;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (uint32_t src = 0; src < kCluster; ++src) {
        const float4 v = ld_dsmem_f32x4(mapa(off, src));
        acc.x += v.x;
        acc.y += v.y;
        acc.z += v.z;
        acc.w += v.w;
      }
      reinterpret_cast<float4*>(out + (size_t)h * kDLat)[d4] = acc;
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
  sparse_attn_kernel<<<rows * kCluster, kAttnThreads, kSmemBytes, s>>>(p);
  return cudaGetLastError();
}

}  // namespace hsa
