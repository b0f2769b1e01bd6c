// sda_scan.cuh -- the index builder's one-CTA scan (with the re-check of
// flagged compressed entries), run by build_scan_kernel (sda_build.cu).
#pragma once

#include <cstdint>

#include "sda_internal.cuh"

namespace sda {

constexpr int kScanThreads = 1024;


// Status bit of one compressed entry (block, slot): 8 = block or slot out of
// its range, 16 = the slot lies past the pool, 0 = good.
__device__ __forceinline__ int32_t entry_bad(int32_t b, int32_t s, int k_per_block,
                                             int64_t swa_pages, int64_t total_pages) {
  if (b < 0 || s < 0 || s >= k_per_block) return 8;
  if (swa_pages + (int64_t)b * k_per_block + s >= total_pages) return 16;
  return 0;
}

// The re-check (one CTA of kScanThreads threads, before the scan): for every
// real token (state_slot >= 0) whose entry range is valid and overlaps a
// flagged slice, OR the bits of its entries into kv_indptr[t + 1] (a length
// becomes -(bits)).  Nothing to do, one pass over the flags, when no slice
// was flagged.  Returns whether a slice was flagged (uniform).
__device__ __forceinline__ bool recheck_entries(int N, int32_t* __restrict__ kv_indptr,
                                                const EntryCheck& ec) {
  __shared__ int s_list[kScanThreads];
  __shared__ int s_n;
  int any = 0;
  for (int b = threadIdx.x; b < ec.n_flags; b += kScanThreads) any |= ec.flags[b];
  if (!__syncthreads_or(any)) return false;
  for (int t0 = 0; t0 < N; t0 += kScanThreads) {
    const int t = t0 + threadIdx.x;
    bool need = false;
    if (t < N && ec.state_slot[t] >= 0) {
      const int32_t c0 = ec.comp_indptr[t], c1 = ec.comp_indptr[t + 1];
      if (c0 >= 0 && c1 > c0 && (int64_t)c1 <= ec.comp_total) {
        const int64_t b0 = ((int64_t)c0 >> 2) / ec.chunks_per_cta;
        const int64_t b1 = ((int64_t)(c1 - 1) >> 2) / ec.chunks_per_cta;
        for (int64_t b = b0; b <= b1 && !need; ++b) need = ec.flags[b] != 0;
      }
    }
    if (threadIdx.x == 0) s_n = 0;
    __syncthreads();
    if (need) s_list[atomicAdd(&s_n, 1)] = t;
    __syncthreads();
    const int n = s_n;
    for (int i = 0; i < n; ++i) {
      const int tt = s_list[i];
      const int32_t c0 = ec.comp_indptr[tt], c1 = ec.comp_indptr[tt + 1];
      int32_t bad = 0;
#pragma unroll 4
      for (int32_t e = c0 + threadIdx.x; e < c1; e += kScanThreads)
        bad |= entry_bad(ec.comp_block[e], ec.comp_slot[e], ec.k_per_block, ec.swa_pages,
                         ec.total_pages);
      const int b8 = __syncthreads_or(bad & 8), b16 = __syncthreads_or(bad & 16);
      if (threadIdx.x == 0 && (b8 || b16)) {
        const int32_t v = kv_indptr[tt + 1];
        kv_indptr[tt + 1] = -((v < 0 ? -v : 0) | (b8 ? 8 : 0) | (b16 ? 16 : 0));
      }
    }
    __syncthreads();  // s_list / s_n are rewritten by the next pass
  }
  return true;
}

// One CTA of kScanThreads threads: the entry re-check above, then an
// in-place inclusive scan of the lengths in
// kv_indptr[1..N] (int64 running total), kv_indptr[0] = 0; negative entries
// are bad tokens (empty slice, their bits OR-ed into *status).  If the total exceeds capacity,
// every slice is emptied and bit 32 is raised.  Writes *status.
__device__ __forceinline__ void build_scan_body(int N, int64_t capacity,
                                                int32_t* __restrict__ kv_indptr,
                                                int32_t* __restrict__ status,
                                                const EntryCheck& ec) {
  // the first lengths are read together with the flags; re-read if the
  // re-check rewrote any
  int32_t first = threadIdx.x < N ? kv_indptr[threadIdx.x + 1] : 0;
  if (recheck_entries(N, kv_indptr, ec)) first = threadIdx.x < N ? kv_indptr[threadIdx.x + 1] : 0;
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
    long long v = t0 == 0 ? first : (t < N ? kv_indptr[t + 1] : 0);
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
