// Compressed-cache write ([890B] §四.1: per-channel softmax gating over the m tokens of a
// group, fp32 for m > 1; [ARCH] §3.2 "Z（压缩权重）的计算": pooling -> RMSNorm -> FP4;
// [890B] §三: main KV E2M1 + scale per 16, indexer K E2M1 + E8M0 per 32; [CED] CSA2: indexer K
// is projected from the main-KV entry).
//
// A persistent CTA of 16 warps writes tiles of 32 entries:
//  1. pooling, one warp per entry (2 per warp), lane l owning channels 16l .. 16l+15: per
//     channel a softmax over the two gate values and the weighted sum of the two wkv values in
//     fp32 (p0 = 1 / (1 + e^(g1 - g0)), x = x1 + p0 (x0 - x1): one exponential and one
//     reciprocal, within a few ulp of x1 of the exact pooled value), then RMSNorm (eps 1e-6,
//     unit gain) as one correctly rounded 1 / rms. The
//     lane's 16 channels are one main-KV group, so its scale (the smallest E8M0 or E4M3 value s
//     with 6 s >= amax, an exact bit computation) and its codes (RNE E2M1 of x / s from the
//     hardware cvt, -0 cleared to +0) come straight from registers; with RoPE, of a copy whose
//     last 64 dims are rotated by the entry's position. The raw inputs of the warp's next
//     entries are loaded while it works;
//  2. the normalised latent is split into three bf16 terms, hi + mid + lo = x exactly (each
//     term the bf16 rounding of what the previous ones left), stacked as the 96 rows (term t,
//     entry r -> row 32 t + r) of one 128B-swizzled K-major tile;
//  3. indexer K^T = W_idx^T . [hi | mid | lo]^T on tcgen05 (kind::f16, bf16 x bf16, fp32
//     accumulate in tensor memory: 128 lanes = K dims, 96 columns), one M=128 N=96 MMA per
//     16-dim k-step, so W_idx is read once per tile. W_idx stays in shared memory for the whole
//     launch as the MN-major A operand; every product is exact and the only roundings are the
//     fp32 accumulations and the final hi + mid + lo sum of the three columns of an entry;
//  4. each warp reads one 32-dim group (its tensor-memory lane quadrant) of 8 entries: the
//     group max is one warp reduction, the E8M0 scale and E2M1 codes follow as in step 1, and
//     the bytes are written in the fragment order of include/hsa.h.
// The accumulators are double-buffered in tensor memory: step 4 of a tile runs while the next
// tile's MMAs (issued as soon as its B tile is written) run into the other buffer.
#include "hsa_common.cuh"
#include "hsa_internal.h"
#include "hsa_tc.cuh"

namespace hsa {
namespace {

constexpr int kWWarps = 16;
constexpr int kWThreads = kWWarps * 32;
constexpr int kTileE = 32;                                 // entries per tile (the MMA's N)
constexpr int kEntPerWarp = kTileE / kWWarps;
constexpr uint32_t kWBytes = (uint32_t)kDLat * kDIdx * 2;  // W_idx, bf16, MN-major A operand
constexpr int kBRows = 3 * kTileE;                         // hi, mid, lo terms of the tile's entries
constexpr uint32_t kBBlock = (uint32_t)kBRows * 128u;      // one 64-dim block of the B tile
constexpr uint32_t kOffW = 0, kOffB = kWBytes, kOffMisc = kOffB + 8 * kBBlock;
constexpr uint32_t kMiscBytes = 64;
constexpr uint32_t kWSmem = kOffMisc + kMiscBytes + 1024;  // + alignment slack
constexpr uint32_t kDCols = 128;                           // columns of one accumulator buffer (96 used)
constexpr uint32_t kTmemCols = 2 * kDCols;                 // two buffers: one computed, one read back
static_assert(kWSmem <= 232448, "shared memory");
static_assert(kEntPerWarp * kWWarps == kTileE, "entries per warp");

// E8M0 byte of the smallest e with 6 * 2^e >= amax (amax >= 0), e clamped to [-127, 127]. With
// amax = f 2^E, f in [1, 2): 6 * 2^(E-2) = 1.5 * 2^E covers f <= 1.5, else 6 * 2^(E-1) does, so
// the byte is the exponent field - 2, + 1 when the mantissa field exceeds half. Zero and
// subnormal amax (< 2^-126 <= 6 * 2^-127) take byte 0.
__device__ __forceinline__ uint32_t e8m0_byte_for(float amax) {
  const uint32_t u = __float_as_uint(amax);
  const int b = (int)(u >> 23) - 2 + ((u & 0x7FFFFFu) > 0x400000u ? 1 : 0);
  return (u >> 23) == 0u ? 0u : (uint32_t)max(0, min(254, b));
}
// 1 / 2^(sb - 127) as two exact power-of-two factors: 2^(127 - sb) and 1 for sb <= 253; for
// sb = 254 (whose inverse is below the normal range) 2^-64 and 2^-63, so (x f1) f2 rounds
// once, exactly like x / s
__device__ __forceinline__ void e8m0_inv(uint32_t sb, float& f1, float& f2) {
  f1 = (sb >= 254u) ? __uint_as_float(63u << 23) : __uint_as_float((254u - sb) << 23);
  f2 = (sb >= 254u) ? __uint_as_float(64u << 23) : 1.f;
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

// 1 / y to within one ulp (rcp.approx; 1 / inf = 0)
__device__ __forceinline__ float rcp_approx(float y) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(y));
  return r;
}

// one E2M1 pair byte (lo -> low nibble), RNE, saturating
__device__ __forceinline__ uint32_t e2m1_pair(float lo, float hi) { return f32x2_to_e2m1x2(hi, lo) & 0xFFu; }
// -0 -> +0 in eight packed E2M1 codes: a nibble keeps its sign bit only if its magnitude bits
// are nonzero (magnitude + 7 carries into bit 3 exactly then; no carry leaves the nibble)
__device__ __forceinline__ uint32_t e2m1_clear_neg_zero(uint32_t w) {
  const uint32_t m = w & 0x77777777u;
  return w & (0x77777777u | ((m + 0x77777777u) & 0x88888888u));
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// bf16x2 of (a, b), round to nearest even; a in the low half
__device__ __forceinline__ uint32_t bf16x2_rn(float a, float b) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
  return r;
}

// RoPE on the main-KV copy of an entry's latent ([ARCH] §3.2 压缩 RoPE, theta = 160000): lane l
// holds dims 16 l .. 16 l + 15, so the rotary dims 448..511 are lanes 28..31, pairs
// (448 + 2k, 449 + 2k) with k = 8 (l - 28) + u. Every lane computes the (cos, sin) of pair
// k = lane: the phase pos * turns[k] wraps modulo one turn exactly in 64-bit integers, and its top
// 24 bits (rounded) give 2 * phase for sincospif, within 2^-23 pi of the exact angle. Lanes 28..31
// then fetch their pairs' values by shuffle. All 32 lanes call it.
__device__ __forceinline__ void rope_rotate16(float (&xm)[16], int64_t pos, int lane, const uint64_t* turns) {
  const uint64_t ph = (uint64_t)pos * turns[lane];
  const float t2 = (float)(uint32_t)((ph + (1ull << 39)) >> 40) * 0x1p-23f;
  float sn, cs;
  sincospif(t2, &sn, &cs);
  const int src0 = (8 * (lane - 28)) & 31;
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const float c = __shfl_sync(0xffffffffu, cs, src0 + u);
    const float sv = __shfl_sync(0xffffffffu, sn, src0 + u);
    if (lane >= 28) {
      const float a = xm[2 * u], b = xm[2 * u + 1];
      xm[2 * u] = fmaf(a, c, -(b * sv));
      xm[2 * u + 1] = fmaf(a, sv, b * c);
    }
  }
}

// (request b, index i) of an entry; entries are numbered request-major
struct Loc {
  int64_t b, i;
};
__device__ __forceinline__ Loc locate(int64_t ge, int64_t n) { return Loc{ge / n, ge % n}; }
// the entry `off` (< 32) places after `base`: one step per request boundary crossed, no division
__device__ __forceinline__ Loc step(Loc base, int off, int64_t n) {
  Loc l{base.b, base.i + off};
  while (l.i >= n) {
    l.i -= n;
    ++l.b;
  }
  return l;
}

// raw inputs of one entry for one lane: per token, its 16 channels of wkv (and of wgate)
template <int kRatio>
struct EntryRaw {
  uint4 kv[kRatio][2];
  uint4 g[kRatio == 2 ? 2 : 1][2];
};

template <int kRatio>
__device__ __forceinline__ void load_entry(const WriteParams& p, bool valid, Loc l, int lane, EntryRaw<kRatio>& r) {
  if (valid) {
    const int64_t tok0 = l.b * p.n_tokens + l.i * kRatio;
#pragma unroll
    for (int tk = 0; tk < kRatio; ++tk) {
      const uint4* src = reinterpret_cast<const uint4*>(p.wkv + (tok0 + tk) * kDLat + 16 * lane);
      r.kv[tk][0] = __ldg(src);
      r.kv[tk][1] = __ldg(src + 1);
      if (kRatio == 2) {
        const uint4* gs = reinterpret_cast<const uint4*>(p.wgate + (tok0 + tk) * kDLat + 16 * lane);
        r.g[tk][0] = __ldg(gs);
        r.g[tk][1] = __ldg(gs + 1);
      }
    }
  } else {
#pragma unroll
    for (int tk = 0; tk < kRatio; ++tk) {
      r.kv[tk][0] = r.kv[tk][1] = make_uint4(0u, 0u, 0u, 0u);
      if (kRatio == 2) r.g[tk][0] = r.g[tk][1] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
}

template <int kRatio>
__global__ void __launch_bounds__(kWThreads, 1) cache_write_kernel(const WriteParams p) {
  extern __shared__ uint8_t wsm_raw[];
  const uint32_t raw_base = smem_u32(wsm_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;     // 1024-byte alignment for the swizzled tiles
  uint8_t* sm = wsm_raw + (base - raw_base);
  const uint32_t sW = base + kOffW, sB = base + kOffB;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(sm + kOffMisc);
  const uint32_t mma_bar = base + kOffMisc + 8u;          // MMAs of the current tile done
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (warp == 0) tmem_alloc(smem_u32(s_tmem), kTmemCols);
  if (tid == 0) {
    mbar_init(mma_bar, 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(s_tmem);
  griddep_wait();
  griddep_launch_dependents();

  const int64_t total = (int64_t)p.batch * p.n_entries;
  const int64_t ntiles = (total + kTileE - 1) / kTileE;
  int64_t tile = blockIdx.x;

  // the warp's first entries go in flight before W_idx is staged
  EntryRaw<kRatio> raw[kEntPerWarp];
  Loc cur = locate(tile * kTileE, p.n_entries);          // first entry of the current tile
#pragma unroll
  for (int j = 0; j < kEntPerWarp; ++j) {
    const int r = kEntPerWarp * warp + j;
    load_entry<kRatio>(p, tile * kTileE + r < total, step(cur, r, p.n_entries), lane, raw[j]);
  }

  // W_idx [512 k][128 d] bf16 -> MN-major 128B-swizzled A operand: 64-dim block mb at mb * 64 KB,
  // row k at k * 128 B, 16-byte chunk (d % 64) / 8 swizzled by k
  for (int i = tid; i < kDLat * kDIdx / 8; i += kWThreads) {
    const int k = i >> 4, c16 = i & 15;
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(p.w_idx) + i);
    sts128(sW + (uint32_t)(c16 >> 3) * 65536u + sw128((uint32_t)k, (uint32_t)(c16 & 7)), v.x, v.y, v.z, v.w);
  }

  const uint32_t idesc = idesc_f16(128, kBRows, true, false, true);
  uint32_t phase = 0;
  // step 4 for tile `etile` (first entry ecur) from the accumulators at column ecol: group
  // q = warp & 3, entries 8 (warp >> 2) .. + 7
  auto epilogue = [&](int64_t etile, Loc ecur, uint32_t ecol) {
    const int q = warp & 3, e0 = 8 * (warp >> 2);
    uint32_t vh[8], vm[8], vl[8];
    const uint32_t ta = tmem + ((uint32_t)(32 * q) << 16) + ecol + (uint32_t)e0;
    TMEM_LD8(ta, vh);
    TMEM_LD8(ta + kTileE, vm);
    TMEM_LD8(ta + 2 * kTileE, vl);
    tmem_wait_ld();
    tmem_regs_ready(vh);
    tmem_regs_ready(vm);
    tmem_regs_ready(vl);
    // the 8 entries as independent chains: value, group max, scale, codes, fragment-order word
    uint32_t word[8], sbs[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float val = (__uint_as_float(vh[j]) + __uint_as_float(vm[j])) + __uint_as_float(vl[j]);
      uint32_t mbits;
      asm("redux.sync.max.u32 %0, %1, 0xffffffff;" : "=r"(mbits) : "r"(__float_as_uint(val) & 0x7FFFFFFFu));
      const uint32_t sb = e8m0_byte_for(__uint_as_float(mbits));
      float f1, f2;
      e8m0_inv(sb, f1, f2);
      // lane 2i builds the byte of dims 2i, 2i+1 of the group
      const float other = __shfl_xor_sync(0xffffffffu, val, 1);
      const uint32_t byte = (lane & 1) ? 0u : e2m1_pair((val * f1) * f2, (other * f1) * f2);
      // fragment order: stored word t of group q (offset 16 t + 4 q) = logical bytes 2t, 2t+1,
      // 8+2t, 9+2t of the group, i.e. the bytes of lanes 4t, 4t+2, 16+4t, 18+4t
      const uint32_t y = byte | (__shfl_down_sync(0xffffffffu, byte, 2) << 8);
      word[j] = e2m1_clear_neg_zero(y | (__shfl_down_sync(0xffffffffu, y, 16) << 16));
      sbs[j] = sb;
    }
    Loc l = step(ecur, e0, p.n_entries);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (etile * kTileE + e0 + j < total) {
        const int64_t entry = (p.start_entry ? __ldg(p.start_entry + l.b) : 0) + l.i;
        if (entry >= 0 && entry < p.cap) {                 // out-of-range entries were flagged in step 1
          const size_t eo = (size_t)l.b * p.cap + entry;
          if (lane < 16 && (lane & 3) == 0) *reinterpret_cast<uint32_t*>(p.ik_q + eo * 64 + 4 * lane + 4 * q) = word[j];
          if (lane == 0) p.ik_s[eo * 4 + q] = (uint8_t)sbs[j];
        }
      }
      if (++l.i == p.n_entries) {
        l.i = 0;
        ++l.b;
      }
    }
  };
  bool mma_ok = true;                 // every MMA-completion wait of this thread succeeded
  int db = 0;                         // accumulator buffer of the tile being computed
  bool have_prev = false;
  int64_t prev_tile = 0;
  Loc prev_cur = cur;
  for (; tile < ntiles; tile += gridDim.x) {
    const Loc nxt = locate((tile + gridDim.x) * kTileE, p.n_entries);
    // ------------------------------------------------------------ 1 + 2: pooling, RMSNorm, main KV, B tile
#pragma unroll
    for (int j = 0; j < kEntPerWarp; ++j) {
      const int r = kEntPerWarp * warp + j;                 // entry row of the tile
      const int64_t ge = tile * kTileE + r;
      float x[16];
      if (kRatio == 1) {
        const uint32_t w[8] = {raw[j].kv[0][0].x, raw[j].kv[0][0].y, raw[j].kv[0][0].z, raw[j].kv[0][0].w,
                               raw[j].kv[0][1].x, raw[j].kv[0][1].y, raw[j].kv[0][1].z, raw[j].kv[0][1].w};
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          x[2 * u] = bf16_lo(w[u]);
          x[2 * u + 1] = bf16_hi(w[u]);
        }
      } else {
        const uint32_t a0[8] = {raw[j].kv[0][0].x, raw[j].kv[0][0].y, raw[j].kv[0][0].z, raw[j].kv[0][0].w,
                                raw[j].kv[0][1].x, raw[j].kv[0][1].y, raw[j].kv[0][1].z, raw[j].kv[0][1].w};
        const uint32_t a1[8] = {raw[j].kv[1][0].x, raw[j].kv[1][0].y, raw[j].kv[1][0].z, raw[j].kv[1][0].w,
                                raw[j].kv[1][1].x, raw[j].kv[1][1].y, raw[j].kv[1][1].z, raw[j].kv[1][1].w};
        const uint32_t g0[8] = {raw[j].g[0][0].x, raw[j].g[0][0].y, raw[j].g[0][0].z, raw[j].g[0][0].w,
                                raw[j].g[0][1].x, raw[j].g[0][1].y, raw[j].g[0][1].z, raw[j].g[0][1].w};
        const uint32_t g1[8] = {raw[j].g[1][0].x, raw[j].g[1][0].y, raw[j].g[1][0].z, raw[j].g[1][0].w,
                                raw[j].g[1][1].x, raw[j].g[1][1].y, raw[j].g[1][1].z, raw[j].g[1][1].w};
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const float x0 = (u & 1) ? bf16_hi(a0[u >> 1]) : bf16_lo(a0[u >> 1]);
          const float x1 = (u & 1) ? bf16_hi(a1[u >> 1]) : bf16_lo(a1[u >> 1]);
          const float q0 = (u & 1) ? bf16_hi(g0[u >> 1]) : bf16_lo(g0[u >> 1]);
          const float q1 = (u & 1) ? bf16_hi(g1[u >> 1]) : bf16_lo(g1[u >> 1]);
          // p0 = 1 / (1 + e^(g1 - g0)) (an infinite power gives p0 = 0), x = x1 + p0 (x0 - x1)
          x[u] = fmaf(rcp_approx(1.f + __expf(q1 - q0)), x0 - x1, x1);
        }
      }
      // the raw registers are free: the warp's entry of the next tile goes in flight
      load_entry<kRatio>(p, (tile + gridDim.x) * kTileE + r < total, step(nxt, r, p.n_entries), lane, raw[j]);

      float ss = 0.f;
#pragma unroll
      for (int u = 0; u < 16; ++u) ss = fmaf(x[u], x[u], ss);
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      const float inv_rms = 1.f / sqrtf(ss / (float)kDLat + 1e-6f);
#pragma unroll
      for (int u = 0; u < 16; ++u) x[u] *= inv_rms;

      if (ge < total) {
        const Loc l = step(cur, r, p.n_entries);
        const int64_t b = l.b, entry = (p.start_entry ? __ldg(p.start_entry + l.b) : 0) + l.i;
        if (entry < 0 || entry >= p.cap) {
          if (lane == 0) flag_status(p.status, HSA_FLAG_WRITE_RANGE);
        } else {
          // main KV: this lane's 16 channels are group `lane`; with RoPE, of the rotated copy
          // (the indexer K below is projected from the latent before RoPE)
          float xm[16];
#pragma unroll
          for (int u = 0; u < 16; ++u) xm[u] = x[u];
          if (p.rope) rope_rotate16(xm, entry, lane, p.rope_turns);
          float amax = 0.f;
#pragma unroll
          for (int u = 0; u < 16; ++u) amax = fmaxf(amax, fabsf(xm[u]));
          uint32_t sb, c8[8];
          if (p.scale_fmt == HSA_SCALE_E8M0) {
            sb = e8m0_byte_for(amax);
            float f1, f2;
            e8m0_inv(sb, f1, f2);
            if (sb < 254u) {                // f2 = 1
#pragma unroll
              for (int u = 0; u < 8; ++u) c8[u] = e2m1_pair(xm[2 * u] * f1, xm[2 * u + 1] * f1);
            } else {
#pragma unroll
              for (int u = 0; u < 8; ++u) c8[u] = e2m1_pair((xm[2 * u] * f1) * f2, (xm[2 * u + 1] * f1) * f2);
            }
          } else {
            sb = e4m3_byte_for(amax);
            const float s = e4m3_to_f32(sb);
#pragma unroll
            for (int u = 0; u < 8; ++u) c8[u] = e2m1_pair(__fdiv_rn(xm[2 * u], s), __fdiv_rn(xm[2 * u + 1], s));
          }
          const size_t eo = (size_t)b * p.cap + entry;
          uint2 codes;
          codes.x = e2m1_clear_neg_zero(c8[0] | (c8[1] << 8) | (c8[2] << 16) | (c8[3] << 24));
          codes.y = e2m1_clear_neg_zero(c8[4] | (c8[5] << 8) | (c8[6] << 16) | (c8[7] << 24));
          *reinterpret_cast<uint2*>(p.kv_q + eo * 256 + 8 * lane) = codes;
          p.kv_s[eo * 32 + lane] = (uint8_t)sb;
        }
      } else {
#pragma unroll
        for (int u = 0; u < 16; ++u) x[u] = 0.f;
      }

      // x = hi + mid + lo exactly, each a bf16; dims 16 lane .. 16 lane + 15 are block lane / 4,
      // 16-byte chunks 2 (lane & 3) and 2 (lane & 3) + 1 of row r
      uint32_t t[3][8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float a = x[2 * u], c = x[2 * u + 1];
        t[0][u] = bf16x2_rn(a, c);
        const float ra = a - bf16_lo(t[0][u]), rc = c - bf16_hi(t[0][u]);
        t[1][u] = bf16x2_rn(ra, rc);
        t[2][u] = bf16x2_rn(ra - bf16_lo(t[1][u]), rc - bf16_hi(t[1][u]));
      }
      // the previous tile's MMAs have finished reading the B tile (waited at its epilogue)
      const uint32_t blk = sB + (uint32_t)(lane >> 2) * kBBlock;
#pragma unroll
      for (int tm = 0; tm < 3; ++tm) {
        const uint32_t row = (uint32_t)(kTileE * tm + r);
        sts128(blk + sw128(row, 2u * (lane & 3)), t[tm][0], t[tm][1], t[tm][2], t[tm][3]);
        sts128(blk + sw128(row, 2u * (lane & 3) + 1u), t[tm][4], t[tm][5], t[tm][6], t[tm][7]);
      }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();

    // ------------------------------------------------------------ 3: K^T = W^T . [hi | mid | lo]^T, 32 k-steps
    // into accumulator buffer db; the previous tile's buffer is read back while these run
    const uint32_t dcol = (uint32_t)db * kDCols;
    if (tid == 0) {
      tc_fence_after();
      const uint64_t a0 = sdesc(sW, 65536u, 1024u), b0 = sdesc(sB, 16u, 1024u);
#pragma unroll
      for (int k = 0; k < kDLat / 16; ++k) {
        const uint32_t ao = ((uint32_t)k * 16u * 128u) >> 4;
        const uint32_t bo = ((uint32_t)(k >> 2) * kBBlock + (uint32_t)(k & 3) * 32u) >> 4;
        umma_f16(tmem + dcol, a0 + ao, b0 + bo, idesc, k > 0);
      }
      umma_commit(mma_bar);
    }
    // ------------------------------------------------------------ 4: the previous tile's indexer K
    if (have_prev) epilogue(prev_tile, prev_cur, dcol ^ kDCols);
    if (!mbar_wait(mma_bar, phase, p.wait_ns)) {
      if (lane == 0) flag_status(p.status, HSA_FLAG_TIMEOUT);
      mma_ok = false;
    }
    phase ^= 1u;
    tc_fence_after();                 // this tile's accumulators (read next iteration) and B tile are done
    prev_tile = tile;
    prev_cur = cur;
    have_prev = true;
    db ^= 1;
    cur = nxt;
  }
  if (have_prev) epilogue(prev_tile, prev_cur, (uint32_t)(db ^ 1) * kDCols);
  // a wait that gave up may have left this CTA's last MMAs running: wait again (bounded) before
  // the tensor memory is freed
  if (__syncthreads_or(!mma_ok) && have_prev && warp == 0) {
    if (!mbar_wait(mma_bar, phase ^ 1u, p.wait_ns) && lane == 0) flag_status(p.status, HSA_FLAG_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_free(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_cache_write(const WriteParams& p, cudaStream_t s) {
  auto kern = (p.ratio == 2) ? cache_write_kernel<2> : cache_write_kernel<1>;
  cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(kern), kWSmem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t ntiles = ((int64_t)p.batch * p.n_entries + kTileE - 1) / kTileE;
  const int grid = (int)imin64(ntiles, (int64_t)sms);
  if (grid < 1) return cudaSuccess;
  return launch_pdl(kern, dim3(grid), dim3(kWThreads), kWSmem, s, p);
}

}  // namespace hsa
