// Compressed-cache write ([890B] §四.1: per-channel softmax gating over the m tokens of a
// group, fp32 for m > 1; [ARCH] §3.2 "Z（压缩权重）的计算": pooling -> RMSNorm -> FP4;
// [890B] §三: main KV E2M1 + scale per 16, indexer K E2M1 + E8M0 per 32; [CED] CSA2: indexer K
// is projected from the main-KV entry).
//
// A persistent CTA handles 16 entries per iteration:
//  1. pooling: one warp per entry; per channel a softmax over the m gate values and the
//     weighted sum of the m wkv values (fp32). Then RMSNorm (eps 1e-6, unit gain), kept in
//     shared memory;
//  2. main-KV quantisation: per 16-channel group, scale = the smallest E8M0 (or E4M3) value
//     s with 6 s >= amax (an exact integer/bit computation); codes are RNE E2M1 of x / s,
//     from the hardware cvt. -0 is cleared to +0;
//  3. indexer K = latent . W_idx (W_idx bf16 kept in shared memory, fp32 FMA), then group-32
//     E8M0 quantisation, written in the fragment byte order of include/hsa.h.
#include "hsa_common.cuh"
#include "hsa_internal.h"

namespace hsa {
namespace {

constexpr int kWThreads = 256;
constexpr int kEnt = 16;
constexpr size_t kOffLat = 0;                                  // [16][512] f32
constexpr size_t kOffW = kOffLat + kEnt * kDLat * 4;          // [512][128] bf16
constexpr size_t kOffK = kOffW + (size_t)kDLat * kDIdx * 2;    // [16][128] f32
constexpr size_t kWSmem = kOffK + kEnt * kDIdx * 4;

// smallest e with 6 * 2^e >= amax (amax > 0), clamped to [-127, 127]; returns the E8M0 byte
__device__ __forceinline__ uint32_t e8m0_byte_for(float amax) {
  if (!(amax > 0.f)) return 0u;
  int E;
  const float m = frexpf(amax, &E);     // amax = m 2^E, m in [0.5, 1)
  int e = (m <= 0.75f) ? E - 3 : E - 2;  // 6 * 2^(E-3) = 0.75 * 2^E
  e = max(-127, min(127, e));
  return (uint32_t)(e + 127);
}

// smallest positive E4M3 value s with 6 s >= amax (saturating at 448); returns the byte
__device__ __forceinline__ uint32_t e4m3_byte_for(float amax) {
  if (!(amax > 6.f * 0.001953125f)) return 1u;          // <= 6 * 2^-9: smallest subnormal
  if (amax > 6.f * 448.f) return 0x7Eu;
  const float t = amax / 6.f;
  uint32_t byte;
  if (t <= 0.015625f) {                                   // subnormal range, steps of 2^-9
    int m = (int)ceilf(t * 512.f);
    byte = (m >= 8) ? (1u << 3) : (uint32_t)m;
  } else {
    int E;
    const float f = frexpf(t, &E);                        // t in [2^(E-1), 2^E)
    int m = (int)ceilf((f * 2.f - 1.f) * 8.f);            // mantissa steps of 1/8
    int ef = E - 1 + 7;
    if (m >= 8) {
      m = 0;
      ++ef;
    }
    byte = ((uint32_t)ef << 3) | (uint32_t)m;
  }
  if (byte > 0x7Eu) byte = 0x7Eu;
  // the fp32 quotient may have rounded down: step up until 6 s >= amax (exact products)
  for (int i = 0; i < 2; ++i)
    if (byte < 0x7Eu && 6.f * e4m3_to_f32(byte) < amax) ++byte;
  return byte;
}

// 16 floats (8 pairs) -> 8 bytes of E2M1 pairs (element 2j low nibble), no -0
__device__ __forceinline__ uint2 pack16(const float* v, float inv_or_s, bool divide) {
  uint32_t b[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float lo = divide ? __fdiv_rn(v[2 * j], inv_or_s) : v[2 * j] * inv_or_s;
    const float hi = divide ? __fdiv_rn(v[2 * j + 1], inv_or_s) : v[2 * j + 1] * inv_or_s;
    uint32_t x = f32x2_to_e2m1x2(hi, lo) & 0xFFu;
    if ((x & 0x07u) == 0u) x &= 0xF0u;
    if ((x & 0x70u) == 0u) x &= 0x0Fu;
    b[j] = x;
  }
  uint2 r;
  r.x = b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24);
  r.y = b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24);
  return r;
}

__device__ __forceinline__ float bf16_to_f32(uint16_t v) { return __uint_as_float((uint32_t)v << 16); }

__global__ void __launch_bounds__(kWThreads, 1) cache_write_kernel(const WriteParams p) {
  extern __shared__ __align__(16) uint8_t wsm[];
  float* lat = reinterpret_cast<float*>(wsm + kOffLat);
  uint16_t* W = reinterpret_cast<uint16_t*>(wsm + kOffW);
  float* Ks = reinterpret_cast<float*>(wsm + kOffK);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  griddep_wait();
  griddep_launch_dependents();

  for (int i = tid; i < kDLat * kDIdx / 8; i += kWThreads)
    reinterpret_cast<uint4*>(W)[i] = __ldg(reinterpret_cast<const uint4*>(p.w_idx) + i);
  __syncthreads();

  const int64_t per_req = p.n_entries;
  const int64_t total = (int64_t)p.batch * per_req;
  const int64_t ntiles = (total + kEnt - 1) / kEnt;
  for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    // ------------------------------------------------------------ 1. pooling + RMSNorm
    for (int el = warp; el < kEnt; el += kWThreads / 32) {
      const int64_t ge = tile * kEnt + el;
      float x[16];
      if (ge < total) {
        const int64_t b = ge / per_req, i = ge % per_req;
        const int64_t tok0 = b * p.n_tokens + i * p.ratio;
        // lane handles channels [8*lane, 8*lane+8) and [256 + 8*lane, ...)
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int c0 = half * 256 + 8 * lane;
          if (p.ratio == 1) {
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(p.wkv + tok0 * kDLat + c0));
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              x[8 * half + 2 * j] = bf16_to_f32((uint16_t)(w[j] & 0xFFFFu));
              x[8 * half + 2 * j + 1] = bf16_to_f32((uint16_t)(w[j] >> 16));
            }
          } else {
            float g[2][8], xv[2][8];
#pragma unroll
            for (int tk = 0; tk < 2; ++tk) {
              const uint4 v = __ldg(reinterpret_cast<const uint4*>(p.wkv + (tok0 + tk) * kDLat + c0));
              const uint4 gg = __ldg(reinterpret_cast<const uint4*>(p.wgate + (tok0 + tk) * kDLat + c0));
              const uint32_t w[4] = {v.x, v.y, v.z, v.w}, wg[4] = {gg.x, gg.y, gg.z, gg.w};
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                xv[tk][2 * j] = bf16_to_f32((uint16_t)(w[j] & 0xFFFFu));
                xv[tk][2 * j + 1] = bf16_to_f32((uint16_t)(w[j] >> 16));
                g[tk][2 * j] = bf16_to_f32((uint16_t)(wg[j] & 0xFFFFu));
                g[tk][2 * j + 1] = bf16_to_f32((uint16_t)(wg[j] >> 16));
              }
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float mx = fmaxf(g[0][j], g[1][j]);
              const float e0 = expf(g[0][j] - mx), e1 = expf(g[1][j] - mx);
              const float s = e0 + e1;
              x[8 * half + j] = (e0 / s) * xv[0][j] + (e1 / s) * xv[1][j];
            }
          }
        }
        float ss = 0.f;
#pragma unroll
        for (int j = 0; j < 16; ++j) ss = fmaf(x[j], x[j], ss);
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        const float rms = sqrtf(ss / (float)kDLat + 1e-6f);
#pragma unroll
        for (int j = 0; j < 16; ++j) x[j] = x[j] / rms;
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) x[j] = 0.f;
      }
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float4* dst = reinterpret_cast<float4*>(lat + el * kDLat + half * 256 + 8 * lane);
        dst[0] = make_float4(x[8 * half], x[8 * half + 1], x[8 * half + 2], x[8 * half + 3]);
        dst[1] = make_float4(x[8 * half + 4], x[8 * half + 5], x[8 * half + 6], x[8 * half + 7]);
      }
    }
    __syncthreads();

    // ------------------------------------------------------------ 2. main-KV quantisation
    for (int gi = tid; gi < kEnt * 32; gi += kWThreads) {
      const int el = gi >> 5, grp = gi & 31;
      const int64_t ge = tile * kEnt + el;
      if (ge >= total) continue;
      const int64_t b = ge / per_req, i = ge % per_req;
      const int64_t entry = (p.start_entry ? __ldg(p.start_entry + b) : 0) + i;
      if (entry < 0 || entry >= p.cap) {
        if (grp == 0) flag_status(p.status, HSA_FLAG_WRITE_RANGE);
        continue;
      }
      const float* v = lat + el * kDLat + grp * 16;
      float amax = 0.f;
#pragma unroll
      for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(v[j]));
      uint32_t sb;
      uint2 codes;
      if (p.scale_fmt == HSA_SCALE_E8M0) {
        sb = e8m0_byte_for(amax);
        const float inv = __uint_as_float((uint32_t)(254 - (int)sb) << 23);   // 2^-(sb-127), exact
        float vv[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) vv[j] = v[j];
        if (sb == 0u || sb == 254u) {
          codes = pack16(vv, e8m0_to_f32(sb), true);
        } else {
          codes = pack16(vv, inv, false);
        }
      } else {
        sb = e4m3_byte_for(amax);
        float vv[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) vv[j] = v[j];
        codes = pack16(vv, e4m3_to_f32(sb), true);
      }
      const size_t eo = (size_t)b * p.cap + entry;
      *reinterpret_cast<uint2*>(p.kv_q + eo * 256 + grp * 8) = codes;
      p.kv_s[eo * 32 + grp] = (uint8_t)sb;
    }

    // ------------------------------------------------------------ 3. indexer projection (fp32)
    {
      const int c = tid & 127, e0 = (tid >> 7) * 8;
      float acc[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] = 0.f;
#pragma unroll 2
      for (int d = 0; d < kDLat; d += 4) {
        const float w0 = bf16_to_f32(W[(d + 0) * kDIdx + c]), w1 = bf16_to_f32(W[(d + 1) * kDIdx + c]);
        const float w2 = bf16_to_f32(W[(d + 2) * kDIdx + c]), w3 = bf16_to_f32(W[(d + 3) * kDIdx + c]);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float4 l = *reinterpret_cast<const float4*>(lat + (e0 + j) * kDLat + d);
          float a = acc[j];
          a = fmaf(l.x, w0, a);
          a = fmaf(l.y, w1, a);
          a = fmaf(l.z, w2, a);
          a = fmaf(l.w, w3, a);
          acc[j] = a;
        }
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) Ks[(e0 + j) * kDIdx + c] = acc[j];
    }
    __syncthreads();
    if (tid < kEnt * 4) {
      const int el = tid >> 2, grp = tid & 3;
      const int64_t ge = tile * kEnt + el;
      if (ge < total) {
        const int64_t b = ge / per_req, i = ge % per_req;
        const int64_t entry = (p.start_entry ? __ldg(p.start_entry + b) : 0) + i;
        if (entry >= 0 && entry < p.cap) {
          const float* v = Ks + el * kDIdx + grp * 32;
          float amax = 0.f;
#pragma unroll
          for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(v[j]));
          const uint32_t sb = e8m0_byte_for(amax);
          float vv[16];
          uint32_t nb[16];
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
            for (int j = 0; j < 16; ++j) vv[j] = v[16 * hh + j];
            uint2 c8 = (sb == 0u || sb == 254u) ? pack16(vv, e8m0_to_f32(sb), true)
                                                : pack16(vv, __uint_as_float((uint32_t)(254 - (int)sb) << 23), false);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              nb[8 * hh + j] = (c8.x >> (8 * j)) & 0xFFu;
              nb[8 * hh + 4 + j] = (c8.y >> (8 * j)) & 0xFFu;
            }
          }
          // fragment order: stored byte 16t + 4grp + {0,1,2,3} = logical 16grp + {2t, 2t+1, 8+2t, 9+2t}
          const size_t eo = (size_t)b * p.cap + entry;
          uint8_t* dst = p.ik_q + eo * 64;
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const uint32_t w = nb[2 * t] | (nb[2 * t + 1] << 8) | (nb[8 + 2 * t] << 16) | (nb[9 + 2 * t] << 24);
            *reinterpret_cast<uint32_t*>(dst + 16 * t + 4 * grp) = w;
          }
          p.ik_s[eo * 4 + grp] = (uint8_t)sb;
        }
      }
    }
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_cache_write(const WriteParams& p, cudaStream_t s) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(cache_write_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kWSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t ntiles = ((int64_t)p.batch * p.n_entries + kEnt - 1) / kEnt;
  int grid = (int)imin64(ntiles, (int64_t)sms);
  if (grid < 1) return cudaSuccess;
  return launch_pdl(cache_write_kernel, dim3(grid), dim3(kWThreads), kWSmem, s, p);
}

}  // namespace hsa
