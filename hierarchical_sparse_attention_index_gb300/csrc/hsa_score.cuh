// Indexer scoring pieces shared by the Full / Reindex scan kernel and the fused Reindex kernel
// (s_t = sum_h w_h ReLU(q_h . k_t), [CED] Figure 5; [ARCH] §3.3):
//  - stage_query: one query's 16 heads x 128 dims to f16 m16n8k16 B fragments in shared memory,
//    after a per-head power-of-two shift that keeps the head's largest |q| in [2^14, 2^15) (exact
//    within f16); the shift is folded back into the head weight;
//  - score_rows32: one warp scores 32 rows of FP4 indexer K held in shared memory in fragment
//    order (include/hsa.h): the hardware E2M1 -> f16x2 convert makes the A operand in registers,
//    each 32-dim group's E8M0 scale is applied exactly in fp32 to its accumulators, and a
//    reduce-scatter over the 4 head lanes leaves lane (g, t) with the score of row 8t + g;
//  - gather_runs: one warp gathers 32 pool slots (four 8-entry runs) of indexer K with cp.async.
#pragma once

#include "hsa_common.cuh"

namespace hsa {

__device__ __forceinline__ uint4 lds128_u(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t lds32_u(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Shared-memory sizes of one staged query: B fragments [2 n-tiles][8 k-steps][32 lanes][2] and
// the 16 shifted head weights.
constexpr int kQFragWords = 2 * 8 * 32 * 2;
constexpr int kQWeights = 16;

// Threads tid < 256 stage the query `q16x128` (bf16 [16 heads][128 dims]) and head weights `w16`
// into `bfrag` / `wsc`; thread tid handles head tid / 16, dims 8 (tid % 16) .. +7. The caller
// synchronises before the fragments are read.
__device__ __forceinline__ void stage_query(const uint16_t* q16x128, const float* w16, uint32_t* bfrag, float* wsc,
                                            int tid) {
  const int h = tid >> 4, d0 = (tid & 15) * 8;
  const uint4 raw = __ldg(reinterpret_cast<const uint4*>(q16x128 + h * kDIdx + d0));
  float x[8];
  const uint32_t rw[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(rw[i] << 16);
    x[2 * i + 1] = __uint_as_float(rw[i] & 0xFFFF0000u);
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
  for (int o = 8; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  int sh = 0;
  if (amax > 0.f) {
    int e;
    frexpf(amax, &e);          // amax = m * 2^e, m in [0.5, 1)
    sh = 15 - e;               // amax * 2^sh in [2^14, 2^15)
  }
  uint32_t pk[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half lo = __float2half_rn(ldexpf(x[2 * i], sh));
    const __half hi = __float2half_rn(ldexpf(x[2 * i + 1], sh));
    pk[i] = (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
  }
  // dims d0..d0+7 -> k-step s = d0/16, t' = (d0%16)/4 and t'+1
  const int ks = d0 >> 4, tp = (d0 & 15) >> 2;
  const int nt = h >> 3, gp = h & 7;
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int ln = 4 * gp + tp + u;
    uint32_t* dst = bfrag + (((size_t)nt * 8 + ks) * 32 + ln) * 2;
    dst[0] = pk[2 * u];
    dst[1] = pk[2 * u + 1];
  }
  if ((tid & 15) == 0) wsc[h] = ldexpf(__ldg(w16 + h), -sh);
}

// The staged query as this lane's MMA B fragments and its 4 head weights (heads 8 nt + 2 t + j).
__device__ __forceinline__ void load_query_frags(const uint32_t* bfrag, const float* wsc, int lane,
                                                 uint32_t (&B)[2][8][2], float (&wr)[2][2]) {
  const int t = lane & 3;
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      const uint2 v = *reinterpret_cast<const uint2*>(bfrag + (((size_t)nt * 8 + s) * 32 + lane) * 2);
      B[nt][s][0] = v.x;
      B[nt][s][1] = v.y;
    }
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int j = 0; j < 2; ++j) wr[nt][j] = wsc[nt * 8 + 2 * t + j];
}

// A warp's 32 rows' E8M0 group scales as floats, once per stage: 2^(b-127) is byte b moved to
// the exponent field (b = 0 only occurs with all-zero codes, where 0 * 0 = 0). `scales` holds 4
// bytes per row; the warp's rows start at row_off; sf_base is the warp's 512-byte area.
__device__ __forceinline__ void stage_group_scales(uint32_t scales, int row_off, uint32_t sf_base, int lane) {
  const uint32_t S = lds32_u(scales + (uint32_t)(row_off + lane) * 4u);
  asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(sf_base + (uint32_t)lane * 16u),
               "r"((S << 23) & 0x7F800000u), "r"((S << 15) & 0x7F800000u), "r"((S << 7) & 0x7F800000u),
               "r"((S >> 1) & 0x7F800000u)
               : "memory");
  __syncwarp();
}

// Scores of the warp's 32 rows (codes: 64 bytes per row in fragment order, rows from row_off).
// Returns the score of row 8t + g (g = lane / 4, t = lane % 4), i.e. the 16-head ReLU-weighted
// sum before any visibility mask. Both 16-row tiles are always scored (their independent chains
// interleave); the caller masks rows that hold no data.
__device__ __forceinline__ float score_rows32(uint32_t codes, int row_off, uint32_t sf_base,
                                              const uint32_t (&B)[2][8][2], const float (&wr)[2][2], int lane) {
  const int g = lane >> 2, t = lane & 3;
  const uint32_t a_base = codes + (uint32_t)(row_off + g) * 64u + 16u * t;
  // vp[mt][0/1]: ReLU-weighted sum over this lane's 4 heads for rows g / g+8 of tile mt
  float vp[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
  for (int mt = 0; mt < 2; ++mt) {
    const uint4 A0 = lds128_u(a_base + (uint32_t)mt * 1024u);
    const uint4 A1 = lds128_u(a_base + (uint32_t)mt * 1024u + 512u);
    const uint4 SF0 = lds128_u(sf_base + (uint32_t)(16 * mt + g) * 16u);
    const uint4 SF1 = lds128_u(sf_base + (uint32_t)(16 * mt + g + 8) * 16u);
    const float sf0[4] = {__uint_as_float(SF0.x), __uint_as_float(SF0.y), __uint_as_float(SF0.z),
                          __uint_as_float(SF0.w)};
    const float sf1[4] = {__uint_as_float(SF1.x), __uint_as_float(SF1.y), __uint_as_float(SF1.z),
                          __uint_as_float(SF1.w)};
    const uint32_t aw0[4] = {A0.x, A0.y, A0.z, A0.w}, aw1[4] = {A1.x, A1.y, A1.z, A1.w};
    // tot[nt][r]: the scaled sums of heads (8 nt + 2 t, +1) for row g (r = 0) or g + 8 (r = 1),
    // packed in pairs
    uint64_t tot[2][2];
#pragma unroll
    for (int gi = 0; gi < 4; ++gi) {
      // group gi = word gi of each row's chunk = k-steps 2gi (bytes 0,1) and 2gi+1 (bytes 2,3)
      uint32_t f0, f1, f2, f3, h0, h1, h2, h3;
      e2m1x8_to_f16x2x4(aw0[gi], f0, f1, f2, f3);
      e2m1x8_to_f16x2x4(aw1[gi], h0, h1, h2, h3);
      const uint64_t sc0 = f2_pack(sf0[gi], sf0[gi]), sc1 = f2_pack(sf1[gi], sf1[gi]);
      float tmp[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        mma_f16_16816_zc(tmp[nt], f0, h0, f1, h1, B[nt][2 * gi][0], B[nt][2 * gi][1]);
        mma_f16_16816(tmp[nt], f2, h2, f3, h3, B[nt][2 * gi + 1][0], B[nt][2 * gi + 1][1]);
      }
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const uint64_t a = f2_pack(tmp[nt][0], tmp[nt][1]), c = f2_pack(tmp[nt][2], tmp[nt][3]);
        tot[nt][0] = gi ? f2_fma(sc0, a, tot[nt][0]) : f2_mul(sc0, a);
        tot[nt][1] = gi ? f2_fma(sc1, c, tot[nt][1]) : f2_mul(sc1, c);
      }
    }
    // ReLU-weighted head sums, the head pair (2t, 2t+1) of each n-tile accumulated as a pair
    uint64_t acc0 = f2_pack(0.f, 0.f), acc1 = acc0;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const uint64_t w2 = f2_pack(wr[nt][0], wr[nt][1]);
      acc0 = f2_fma(w2, f2_relu(tot[nt][0]), acc0);
      acc1 = f2_fma(w2, f2_relu(tot[nt][1]), acc1);
    }
    float lo, hi;
    f2_unpack(acc0, lo, hi);
    vp[mt][0] = lo + hi;
    f2_unpack(acc1, lo, hi);
    vp[mt][1] = lo + hi;
  }
  // Reduce-scatter over the 4 head lanes t of a row group: after it, lane (g, t) holds the full
  // 16-head score of row 8t + g of the warp (tile t >> 1, row g + 8 (t & 1)).
  const bool hi2 = (t & 2) != 0, hi1 = (t & 1) != 0;
  const float k0 = (hi2 ? vp[1][0] : vp[0][0]) + __shfl_xor_sync(0xffffffffu, hi2 ? vp[0][0] : vp[1][0], 2);
  const float k1 = (hi2 ? vp[1][1] : vp[0][1]) + __shfl_xor_sync(0xffffffffu, hi2 ? vp[0][1] : vp[1][1], 2);
  return (hi1 ? k1 : k0) + __shfl_xor_sync(0xffffffffu, hi1 ? k0 : k1, 1);
}

// One warp gathers its 32 pool slots (lane l holds slot l's pool value pv): run u (slots
// 8u .. 8u+7) covers the 8-position block its first (else its last) slot names (a run may start
// with empty slots: a window block of the pool tail keeps only its newest positions) and is fetched
// (64-byte codes of 8 entries and their 4-byte scales, with cp.async, into dc / ds) only if that
// block is in range; slot l is scored (slots[l] = its position) only if it holds
// block + l % 8 and is visible, else slots[l] = -1; anything inconsistent is flagged. Ends with
// a commit.
template <bool kPoolTail>
__device__ __forceinline__ void gather_runs(const uint8_t* ik_q, const uint8_t* ik_s, int64_t ebase, int64_t cap,
                                            int vis, int pv, int lane, uint32_t dc, uint32_t ds, int* slots,
                                            uint32_t* status) {
  const int j = lane & 7;
  // the run's block: its first slot's position or, with a pool tail, when that slot is empty
  // (only the first window block starts with empty slots, and its last slot is live), its last
  // slot's position - 7
  const int v0 = __shfl_sync(0xffffffffu, pv, lane & ~7);
  int base = v0;
  if (kPoolTail) {
    const int v7 = __shfl_sync(0xffffffffu, pv, lane | 7);
    base = v0 >= 0 ? v0 : (v7 >= 0 ? v7 - 7 : -1);
  }
  const bool bok = (base >= 0) && ((base & 7) == 0) && (base < cap);
  int outv = -1;
  if (bok && pv >= 0) {
    if (pv == base + j && pv < vis) outv = pv;
    else if (pv != base + j || pv >= cap) flag_status(status, HSA_FLAG_INDEX_RANGE);
  } else if (j == 0 && base >= 0 && !bok) {
    flag_status(status, HSA_FLAG_INDEX_RANGE);
  }
  slots[lane] = outv;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int bb = __shfl_sync(0xffffffffu, base, 8 * u);
    if (bb >= 0 && (bb & 7) == 0 && bb < cap) cp_async16(dc + u * 512 + lane * 16, ik_q + (ebase + bb) * 64 + lane * 16);
  }
  const int us = (lane >> 1) & 3;
  const int bs = __shfl_sync(0xffffffffu, base, 8 * us);
  if (lane < 8 && bs >= 0 && (bs & 7) == 0 && bs < cap)
    cp_async16(ds + us * 32 + (lane & 1) * 16, ik_s + (ebase + bs) * 4 + (lane & 1) * 16);
  cp_async_commit();
}

}  // namespace hsa
