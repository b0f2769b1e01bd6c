// sda_scan.cuh -- the index builder's one-CTA scan, shared by its own kernel
// (sda_build.cu) and by the fused scan + work-plan kernel (sda_plan.cu).
#pragma once

#include <cstdint>

namespace sda {

constexpr int kScanThreads = 1024;

// One CTA of kScanThreads threads: in-place inclusive scan of the lengths in
// kv_indptr[1..N] (int64 running total), kv_indptr[0] = 0; negative entries
// are bad tokens (empty slice, their bits OR-ed into *status).  If the total exceeds capacity,
// every slice is emptied and bit 32 is raised.  Writes *status.
__device__ __forceinline__ void build_scan_body(int N, int64_t capacity,
                                                int32_t* __restrict__ kv_indptr,
                                                int32_t* __restrict__ status) {
  __shared__ long long warp_sums[32];
  __shared__ long long s_carry;
  __shared__ int s_over;
  __shared__ int s_flags;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    s_carry = 0;
    s_over = 0;
    s_flags = 0;
  }
  __syncthreads();
  for (int t0 = 0; t0 < N; t0 += kScanThreads) {
    const int t = t0 + threadIdx.x;
    long long v = t < N ? kv_indptr[t + 1] : 0;
    if (v < 0) {
      atomicOr(&s_flags, (int)(-v));
      v = 0;
    }
    long long x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      long long y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
      long long w = warp_sums[lane], s = w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        long long y = __shfl_up_sync(0xffffffffu, s, o);
        if (lane >= o) s += y;
      }
      warp_sums[lane] = s - w;
    }
    __syncthreads();
    const long long incl = s_carry + warp_sums[warp] + x;
    if (t < N) {
      if (incl > capacity) s_over = 1;
      kv_indptr[t + 1] = (int32_t)(incl > capacity ? capacity : incl);
    }
    __syncthreads();
    if (threadIdx.x == kScanThreads - 1) s_carry = incl;
    __syncthreads();
  }
  if (threadIdx.x == 0) kv_indptr[0] = 0;
  __syncthreads();
  if (s_over)
    for (int t = threadIdx.x; t <= N; t += kScanThreads) kv_indptr[t] = 0;
  if (threadIdx.x == 0) *status = s_flags | (s_over ? 32 : 0);
}

}  // namespace sda
