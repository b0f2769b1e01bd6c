// sda_topk.cu -- top-k selection of compressed-cache entries straight into the
// slot lists the index builder consumes: for every token, the k best-scored
// of its candidate positions, emitted in position order as (block id, slot in
// block) pairs through the token's block table.
//
// Source: the sglang attention tag page, entry "DSV4.1 新增索引器内核，重做 Top-K
// v2 分派": padding is NaN, not a very small number, so that a legitimate -inf
// stays selectable; the page-table transform is a separate step from the
// selection.  The pool entry of a compressed position is block_id *
// K_PER_BLOCK + slot_in_block (the paged_decode.py docstring on the PR 28392
// page), which sda_build_indices then offsets by swa_pages.
//
// Order used (plainest reading, identical on both sides of the parity tests):
// larger score first, -0 equal to +0, NaN below -inf, equal scores by
// increasing position.  Scores map to 32-bit keys that preserve that order,
// so the selection is an exact radix select on integers:
//   1. topk_indptr_kernel (one CTA): comp_indptr = prefix sums of min(k, n_t)
//      (for batches of up to 4096 tokens each select CTA computes its own
//      entry instead, and this launch is skipped);
//   2. topk_select_kernel (one CTA per token): up to three digit passes
//      (MSB first) find the key T of the k-th best candidate and how many
//      candidates equal to T to keep (stopping early once the digit bin that
//      holds the k-th key is kept whole); one ordered pass then keeps every
//      key above T and the first `need` keys equal to T, writing each kept
//      position at its rank among kept positions (a block scan per chunk), so
//      the output is in increasing position with no sort.
// A token's keys are staged once in shared memory when its row fits
// (<= kSmemKeys candidates); longer rows are re-read from global memory (L2)
// by each pass.  Digits are 11, 11 and 10 bits wide: the leading bits of real
// scores (sign and exponent) crowd into few values, and wide first digits
// leave the threshold bin small, so the passes usually stop after the second.
#include <cuda_runtime.h>

#include <cstdint>

#include "sda_internal.cuh"

namespace sda {

namespace {

constexpr int kTopkThreads = 1024;
constexpr int kSmemKeys = 9216;  // 36 KB of staged keys (static shared memory <= 48 KB)
constexpr int kBins = 2048;      // digit histogram (11-bit digits)
static_assert(kBins == 2 * kTopkThreads, "two histogram bins per thread");

__device__ __forceinline__ uint32_t score_key(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7fffffffu) > 0x7f800000u) return 0u;  // NaN: below every number
  if (u == 0x80000000u) u = 0u;                     // -0 ranks as +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ int valid_length(const int32_t* lengths, int t, int64_t stride) {
  const int n = lengths[t];
  return (n < 0 || n > stride) ? 0 : n;
}

// Exclusive block scan of one 32-bit value per thread (blockDim.x == kTopkThreads);
// *total receives the block sum.  `warp_sums` holds kTopkThreads / 32 words.
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t* warp_sums,
                                                         uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    constexpr int kWarps = kTopkThreads / 32;
    uint32_t w = lane < kWarps ? warp_sums[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < kWarps) warp_sums[lane] = w;  // inclusive prefix of the warp totals
  }
  __syncthreads();
  const uint32_t before = warp == 0 ? 0u : warp_sums[warp - 1];
  *total = warp_sums[kTopkThreads / 32 - 1];
  __syncthreads();  // warp_sums is reused by the next call
  return before + x - v;
}

// comp_indptr[0..N] = prefix sums of min(k, n_t); bit 1 for a bad length, bit 32
// (and every list empty) if the total exceeds capacity.
__global__ void __launch_bounds__(kTopkThreads) topk_indptr_kernel(
    const int32_t* __restrict__ lengths, int64_t score_stride, int N, int k, int64_t capacity,
    int32_t* __restrict__ comp_indptr, int32_t* __restrict__ status) {
  pdl_wait();
  __shared__ uint32_t warp_sums[kTopkThreads / 32];
  __shared__ int s_flags;
  if (threadIdx.x == 0) s_flags = 0;
  __syncthreads();
  // First pass: the total (to check capacity); second pass: the prefix sums.
  uint64_t total = 0;
  for (int base = 0; base < N; base += kTopkThreads) {
    const int t = base + threadIdx.x;
    uint32_t c = 0;
    if (t < N) {
      const int n = lengths[t];
      if (n < 0 || n > score_stride) atomicOr(&s_flags, 1);
      const int vn = valid_length(lengths, t, score_stride);
      c = static_cast<uint32_t>(vn < k ? vn : k);
    }
    uint32_t chunk;
    block_exclusive_scan(c, warp_sums, &chunk);
    total += chunk;
  }
  const bool over = total > static_cast<uint64_t>(capacity);
  uint32_t run = 0;
  if (threadIdx.x == 0) comp_indptr[0] = 0;
  for (int base = 0; base < N; base += kTopkThreads) {
    const int t = base + threadIdx.x;
    uint32_t c = 0;
    if (t < N && !over) {
      const int vn = valid_length(lengths, t, score_stride);
      c = static_cast<uint32_t>(vn < k ? vn : k);
    }
    uint32_t chunk;
    const uint32_t ex = block_exclusive_scan(c, warp_sums, &chunk);
    if (t < N) comp_indptr[t + 1] = static_cast<int32_t>(run + ex + c);
    run += chunk;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const int f = s_flags | (over ? 32 : 0);
    if (f) atomicOr(status, f);
  }
  pdl_trigger();
}

// Each thread handles groups of kIpt consecutive positions (one 16-byte
// shared-memory access for staged keys), so that the histogram passes and
// the ordered pass take a quarter of the loop trips and block scans.
constexpr int kIpt = 4;

// Sum over the block of two values per thread (FUSED offsets).
__device__ __forceinline__ void block_sum2(uint32_t a, uint32_t b, uint32_t* sa, uint32_t* sb,
                                           uint32_t (*parts)[2]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  a = __reduce_add_sync(0xffffffffu, a);
  b = __reduce_add_sync(0xffffffffu, b);
  if (lane == 0) parts[warp][0] = a, parts[warp][1] = b;
  __syncthreads();
  uint32_t x = 0, y = 0;
  for (int w = 0; w < kTopkThreads / 32; ++w) x += parts[w][0], y += parts[w][1];
  *sa = x;
  *sb = y;
  __syncthreads();
}

// FUSED (batches of at most kFusedTokens tokens whose kept counts sum below
// 2^31): each CTA also sums the kept counts of the tokens before it and of
// all tokens (lengths are a few KB, read from L2 by every CTA), writes its own
// comp_indptr entry and checks the capacity, which saves the separate scan
// launch.
constexpr int kFusedTokens = 4096;

template <bool STAGED, bool FUSED>
__global__ void __launch_bounds__(kTopkThreads, 2) topk_select_kernel(
    const float* __restrict__ scores, int64_t score_stride, const int32_t* __restrict__ lengths,
    const int32_t* __restrict__ block_table, int64_t bt_stride, int N, int k, int k_per_block,
    int64_t capacity, int32_t* __restrict__ comp_indptr, int32_t* __restrict__ comp_block,
    int32_t* __restrict__ comp_slot, int32_t* __restrict__ status) {
  pdl_wait();
  __shared__ __align__(16) uint32_t s_keys[STAGED ? kSmemKeys : kIpt];
  __shared__ uint32_t hist[kBins];
  __shared__ uint32_t warp_sums[kTopkThreads / 32];
  __shared__ uint32_t parts[FUSED ? kTopkThreads / 32 : 1][2];
  __shared__ uint32_t s_digit, s_above, s_count;
  const int t = blockIdx.x;
  const int tid = threadIdx.x;
  const int n = valid_length(lengths, t, score_stride);
  const int kk = n < k ? n : k;
  int32_t out0;
  if constexpr (FUSED) {
    uint32_t before = 0, all = 0;
    int bad = 0;
    for (int u = tid; u < N; u += kTopkThreads) {
      const int lu = lengths[u];
      bad |= (lu < 0 || lu > score_stride) ? 1 : 0;
      const int vu = (lu < 0 || lu > score_stride) ? 0 : lu;
      const uint32_t c = static_cast<uint32_t>(vu < k ? vu : k);
      all += c;
      before += u < t ? c : 0u;
    }
    bad = __syncthreads_or(bad);
    uint32_t s_before, s_all;
    block_sum2(before, all, &s_before, &s_all, parts);
    const bool over = static_cast<int64_t>(s_all) > capacity;
    if (tid == 0) {
      comp_indptr[t + 1] = over ? 0 : static_cast<int32_t>(s_before + kk);
      if (t == 0) {
        comp_indptr[0] = 0;
        const int f = (bad ? 1 : 0) | (over ? 32 : 0);
        if (f) atomicOr(status, f);
      }
    }
    if (over || kk == 0) return;
    out0 = static_cast<int32_t>(s_before);
  } else {
    out0 = comp_indptr[t];
    // kk == 0, or the lists were emptied for lack of capacity
    if (kk == 0 || comp_indptr[t + 1] - out0 != kk) return;
  }
  const float* row = scores + static_cast<size_t>(t) * score_stride;
  const int32_t* bt = block_table + static_cast<size_t>(t) * bt_stride;
  const int groups = (n + kIpt - 1) / kIpt;
  int flags = 0;

  auto emit = [&](int idx, int p) {
    const int32_t blk = bt[p / k_per_block];
    if (blk < 0) flags |= 4;
    comp_block[out0 + idx] = blk;
    comp_slot[out0 + idx] = p % k_per_block;
  };
  // The keys of positions kIpt*g .. kIpt*g+kIpt-1 (0 past the row's end;
  // `valid` tells them apart from NaN keys).
  auto keys_at = [&](int g, uint32_t (&key)[kIpt]) {
    if (STAGED) {
      const uint4 v = reinterpret_cast<const uint4*>(s_keys)[g];
      key[0] = v.x, key[1] = v.y, key[2] = v.z, key[3] = v.w;
    } else {
#pragma unroll
      for (int e = 0; e < kIpt; ++e) {
        const int p = kIpt * g + e;
        key[e] = p < n ? score_key(__ldg(row + p)) : 0u;
      }
    }
  };

  bool nan_seen = false;
  if (kk == n) {  // every candidate is kept, in position order
    for (int p = tid; p < n; p += kTopkThreads) {
      nan_seen |= score_key(row[p]) == 0u;
      emit(p, p);
    }
  } else {
    if (STAGED) {
      for (int g = tid; g < groups; g += kTopkThreads) {
        uint32_t key[kIpt];
#pragma unroll
        for (int e = 0; e < kIpt; ++e) {
          const int p = kIpt * g + e;
          key[e] = p < n ? score_key(row[p]) : 0u;
          nan_seen |= p < n && key[e] == 0u;
        }
        reinterpret_cast<uint4*>(s_keys)[g] = make_uint4(key[0], key[1], key[2], key[3]);
      }
      __syncthreads();
    }
    // Digits of 11, 11 and 10 bits (MSB first): bins 2047 - 2i and 2046 - 2i
    // belong to thread i for the suffix sums.
    uint32_t prefix = 0, mask = 0, need = static_cast<uint32_t>(kk);
#pragma unroll 1
    for (int pass = 0; pass < 3; ++pass) {
      const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
      const uint32_t dmask = pass == 2 ? 0x3ffu : 0x7ffu;
      for (int b = tid; b < kBins; b += kTopkThreads) hist[b] = 0;
      __syncthreads();
      for (int g = tid; g < groups; g += kTopkThreads) {
        uint32_t key[kIpt];
        keys_at(g, key);
#pragma unroll
        for (int e = 0; e < kIpt; ++e) {
          const bool valid = kIpt * g + e < n;
          if (!STAGED && pass == 0) nan_seen |= valid && key[e] == 0u;
          if (valid && (key[e] & mask) == prefix) atomicAdd(&hist[(key[e] >> shift) & dmask], 1u);
        }
      }
      __syncthreads();
      const uint32_t hi = hist[kBins - 1 - 2 * tid], lo = hist[kBins - 2 - 2 * tid];
      uint32_t total;
      const uint32_t above = block_exclusive_scan(hi + lo, warp_sums, &total);  // keys in higher bins
      if (above < need && above + hi >= need) {
        s_digit = kBins - 1 - 2 * tid;
        s_above = above;
        s_count = hi;
      } else if (above + hi < need && above + hi + lo >= need) {
        s_digit = kBins - 2 - 2 * tid;
        s_above = above + hi;
        s_count = lo;
      }
      __syncthreads();
      prefix |= s_digit << shift;
      mask |= dmask << shift;
      need -= s_above;
      const bool whole_bin = need == s_count;  // every key of the bin is kept: done
      __syncthreads();
      if (whole_bin) break;
    }
    // Keep every key whose leading (mask) bits exceed prefix, and the first
    // `need` keys whose leading bits equal it (with the full mask: the k-th
    // best key T itself), each at its rank among the kept positions.
    uint32_t kept = 0, ties = 0;
    for (int g0 = 0; g0 < groups; g0 += kTopkThreads) {
      const int g = g0 + tid;
      uint32_t key[kIpt] = {0u, 0u, 0u, 0u};
      if (g < groups) keys_at(g, key);
      uint32_t gt_bits = 0, eq_bits = 0;
#pragma unroll
      for (int e = 0; e < kIpt; ++e) {
        const bool valid = g < groups && kIpt * g + e < n;
        const uint32_t m = key[e] & mask;
        gt_bits |= (valid && m > prefix) ? 1u << e : 0u;
        eq_bits |= (valid && m == prefix) ? 1u << e : 0u;
      }
      uint32_t tot;
      const uint32_t ex =
          block_exclusive_scan((static_cast<uint32_t>(__popc(eq_bits)) << 16) | __popc(gt_bits),
                               warp_sums, &tot);
      const uint32_t room = need > ties ? need - ties : 0u;  // ties still to keep
      uint32_t gt_before = ex & 0xffffu, eq_before = ex >> 16;
#pragma unroll
      for (int e = 0; e < kIpt; ++e) {
        const bool gt = (gt_bits >> e) & 1u, eq = (eq_bits >> e) & 1u;
        if (gt || (eq && eq_before < room))
          emit(static_cast<int>(kept + gt_before + min(eq_before, room)), kIpt * g + e);
        gt_before += gt;
        eq_before += eq;
      }
      const uint32_t gt_tot = tot & 0xffffu, eq_tot = tot >> 16;
      kept += gt_tot + min(eq_tot, room);
      ties += eq_tot;
    }
  }
  if (nan_seen) flags |= 8;
  if (__syncthreads_or(flags)) {
    if (flags) atomicOr(status, flags);
  }
  pdl_trigger();
}

}  // namespace

cudaError_t launch_topk_slots(const float* scores, int64_t score_stride, const int32_t* lengths,
                              const int32_t* block_table, int64_t bt_stride, int N, int k,
                              int k_per_block, int32_t* comp_indptr, int32_t* comp_block,
                              int32_t* comp_slot, int64_t capacity, int32_t* status,
                              cudaStream_t st) {
  const int64_t max_keep = k < score_stride ? k : score_stride;
  const bool fused = N > 0 && N <= kFusedTokens && k > 0 && N * max_keep < (int64_t{1} << 31);
  if (!fused) {
    cudaError_t e = launch_pdl(topk_indptr_kernel, dim3(1), dim3(kTopkThreads), 0, st, lengths,
                               score_stride, N, k, capacity, comp_indptr, status);
    if (e != cudaSuccess || N == 0 || k == 0) return e;
  }
  const bool staged = score_stride <= kSmemKeys;
#define SDA_TOPK(S, F)                                                                    \
  launch_pdl(topk_select_kernel<S, F>, dim3(N), dim3(kTopkThreads), 0, st, scores,      \
             score_stride, lengths, block_table, bt_stride, N, k, k_per_block, capacity, \
             comp_indptr, comp_block, comp_slot, status)
  if (fused) return staged ? SDA_TOPK(true, true) : SDA_TOPK(false, true);
  return staged ? SDA_TOPK(true, false) : SDA_TOPK(false, false);
#undef SDA_TOPK
}

}  // namespace sda
