// Device helpers shared by the score kernels: a block exclusive scan and the histogram
// threshold search behind the exact top-k selection.
#pragma once

#include "hsa_common.cuh"
#include "hsa_internal.h"

namespace hsa {

// Exclusive prefix sum over the first `nthreads` threads (a multiple of 32); scratch holds 32 ints.
// The caller's threads must all call it (named barrier `bar_id` over `nthreads`).
__device__ __forceinline__ int excl_scan(int v, int* scratch, int bar_id, int nthreads, int* total, int tid = -1) {
  if (tid < 0) tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scratch[warp] = x;
  named_bar_sync(bar_id, nthreads);
  const int nw = nthreads >> 5;
  if (warp == 0) {
    int t = (lane < nw) ? scratch[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    if (lane < nw) scratch[lane] = t;   // inclusive warp totals
  }
  named_bar_sync(bar_id, nthreads);
  const int before = (warp > 0) ? scratch[warp - 1] : 0;
  *total = scratch[nw - 1];
  named_bar_sync(bar_id, nthreads);
  return before + x - v;
}

// Threshold bin of a top-K over a 4096-bin histogram in shared memory held by NT threads (thread 0
// holding the highest bins): the bin holding the K-th largest key and the count above it go to
// out[0], out[1]; -1 and the total when the histogram holds K or fewer. Returns the total. All
// NT threads call it (named barrier 1).
template <int NT>
__device__ __forceinline__ int smem_threshold(const uint32_t* hist, int K, int* scratch, int* out, int tid) {
  constexpr int kPer = kHistBins / NT;
  const int top = kHistBins - kPer * (tid + 1);
  int hc[kPer], local = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    hc[i] = (int)hist[top + i];
    local += hc[i];
  }
  int total;
  const int excl = excl_scan(local, scratch, 1, NT, &total, tid);
  if (total <= K) {
    if (tid == 0) {
      out[0] = -1;
      out[1] = total;
    }
  } else if (excl < K && excl + local >= K) {
    int run = excl;
#pragma unroll
    for (int i = kPer - 1; i >= 0; --i) {
      if (run + hc[i] >= K) {
        out[0] = top + i;
        out[1] = run;
        break;
      }
      run += hc[i];
    }
  }
  named_bar_sync(1, NT);
  return total;
}

}  // namespace hsa
