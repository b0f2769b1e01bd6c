// sda_plan.cu -- device-side work planning (split-L) and the log-sum-exp
// combine of split tokens.
//
// The plan runs on the device because kv_indptr lives there and the decode
// call must stay capturable in a CUDA graph (the reason the paged_decode.py
// docstring gives for the whole design: no per-forward shape that depends on
// host-side lengths).  Splitting long lists and merging the pieces is not on
// the page; it is how the hot path fills all SMs when tokens are few or
// lists are long.
#include <cuda_bf16.h>

#include "sda_internal.cuh"
#include "sda_scan.cuh"

namespace sda {

namespace {

constexpr int kPlanThreads = 1024;
constexpr int kBuckets = 33;  // bucket b holds units of length in [2^(b-1), 2^b); 0 = empty

__device__ __forceinline__ int len_bucket(int len) { return len <= 0 ? 0 : 32 - __clz(len); }

// Exclusive block-wide scan of one int per thread (1024 threads); returns the
// prefix and stores the block total in *total (smem scratch of 32 ints).
__device__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = warp_sums[lane];
    int s = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    warp_sums[lane] = s - w;  // exclusive warp offsets
    if (lane == 31) *total = s;
  }
  __syncthreads();
  const int r = warp_sums[warp] + x - v;
  __syncthreads();
  return r;
}

struct TokenSplit {
  int len, pieces, piece_len;
};

__device__ __forceinline__ TokenSplit token_split(const int32_t* indptr, int t, int chunk, int tile) {
  TokenSplit s;
  int L = indptr[t + 1] - indptr[t];
  s.len = L > 0 ? L : 0;
  s.pieces = s.len == 0 ? 1 : (s.len + chunk - 1) / chunk;
  const int even = (s.len + s.pieces - 1) / s.pieces;
  s.piece_len = s.pieces == 1 ? s.len : ((even + tile - 1) / tile) * tile;
  return s;
}

__device__ __forceinline__ void plan_body(const int32_t* __restrict__ indptr, int N,
                                          long long total_indices, int hg, int grid, int tile,
                                          int min_chunk, WsHeader* __restrict__ hdr,
                                          int4* __restrict__ units, int4* __restrict__ splits) {
  __shared__ int warp_sums[32];
  __shared__ int s_total[2];
  __shared__ int bucket_count[kBuckets];
  __shared__ int bucket_cursor[kBuckets];
  __shared__ int s_chunk;

  if (threadIdx.x < kBuckets) bucket_count[threadIdx.x] = 0;
  __syncthreads();
  // kv_indptr must be a true prefix sum inside [0, total_indices]; otherwise
  // nothing is planned (out is left unwritten) and the error word reads 2, so
  // that no kernel ever reads kv_indices out of bounds.
  int bad = 0;
  for (int t = threadIdx.x; t <= N; t += kPlanThreads) {
    const int v = indptr[t];
    if (v < 0 || (long long)v > total_indices || (t < N && indptr[t + 1] < v)) bad = 1;
  }
  if (__syncthreads_or(bad)) {
    if (threadIdx.x == 0) {
      hdr->n_units = 0;
      hdr->n_split = 0;
      hdr->n_parts = 0;
      hdr->chunk = 0;
      hdr->error = 2;
    }
    return;
  }
  if (threadIdx.x == 0) {
    long long T = N > 0 ? (long long)indptr[N] - (long long)indptr[0] : 0;
    if (T < 0) T = 0;
    long long target = (T * hg + grid - 1) / grid;
    // a multiple of the tile, so that every piece but the last is whole
    // tiles and no piece is empty
    long long chunk = ((target + tile - 1) / tile) * tile;
    if (chunk < min_chunk) chunk = min_chunk;
    if (chunk > (1ll << 30)) chunk = 1ll << 30;
    s_chunk = (int)chunk;
  }
  __syncthreads();
  const int chunk = s_chunk;

  // pass 1: unit counts per length bucket
  for (int t0 = 0; t0 < N; t0 += kPlanThreads) {
    const int t = t0 + threadIdx.x;
    if (t < N) {
      TokenSplit s = token_split(indptr, t, chunk, tile);
      for (int k = 0; k < s.pieces; ++k) {
        int plen = s.pieces == 1 ? s.len : min(s.piece_len, s.len - k * s.piece_len);
        atomicAdd(&bucket_count[len_bucket(plen)], hg);
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int b = kBuckets - 1; b >= 0; --b) {  // longest pieces first
      bucket_cursor[b] = acc;
      acc += bucket_count[b];
    }
    hdr->n_units = acc;
  }
  __syncthreads();

  // pass 2: emit units, partial rows and the split list
  int part_carry = 0, split_carry = 0;
  for (int t0 = 0; t0 < N; t0 += kPlanThreads) {
    const int t = t0 + threadIdx.x;
    TokenSplit s{0, 1, 0};
    if (t < N) s = token_split(indptr, t, chunk, tile);
    const bool split = t < N && s.pieces > 1;
    const int part_base = block_exclusive_scan(split ? s.pieces : 0, warp_sums, &s_total[0]) + part_carry;
    const int split_idx = block_exclusive_scan(split ? 1 : 0, warp_sums, &s_total[1]) + split_carry;
    if (t < N) {
      const int begin = indptr[t];
      for (int k = 0; k < s.pieces; ++k) {
        const int plen = s.pieces == 1 ? s.len : min(s.piece_len, s.len - k * s.piece_len);
        const int pos = atomicAdd(&bucket_cursor[len_bucket(plen)], hg);
        const int row = split ? part_base + k : -1;
        for (int g = 0; g < hg; ++g)
          units[pos + g] = make_int4(t, begin + k * s.piece_len, plen, make_unit_meta(g, row));
      }
      if (split) splits[split_idx] = make_int4(t, part_base, s.pieces, 0);
    }
    part_carry += s_total[0];
    split_carry += s_total[1];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    hdr->n_split = split_carry;
    hdr->n_parts = part_carry;
    hdr->chunk = chunk;
    hdr->error = 0;
  }
}

__global__ void __launch_bounds__(kPlanThreads)
plan_kernel(const int32_t* __restrict__ indptr, int N, long long total_indices, int hg, int grid,
            int tile, int min_chunk, WsHeader* __restrict__ hdr, int4* __restrict__ units,
            int4* __restrict__ splits) {
  pdl_wait();
  pdl_trigger();
  plan_body(indptr, N, total_indices, hg, grid, tile, min_chunk, hdr, units, splits);
}

// The index builder's scan and the plan in one CTA (sda_build_decode): the
// scan turns the per-token lengths into kv_indptr, and the plan reads it
// straight back, which saves the plan's own launch.
static_assert(kPlanThreads == kScanThreads, "one CTA runs both bodies");
__global__ void __launch_bounds__(kPlanThreads)
scan_plan_kernel(int N, int64_t capacity, int32_t* __restrict__ kv_indptr,
                 int32_t* __restrict__ status, int hg, int grid, int tile, int min_chunk,
                 WsHeader* __restrict__ hdr, int4* __restrict__ units, int4* __restrict__ splits) {
  pdl_wait();
  pdl_trigger();
  build_scan_body(N, capacity, kv_indptr, status);
  __syncthreads();  // kv_indptr is final (this CTA wrote it)
  plan_body(kv_indptr, N, (long long)capacity, hg, grid, tile, min_chunk, hdr, units, splits);
}

// Merge the pieces of each split token:
//   M   = max(sink*log2e, max_k m_k)
//   out = sum_k 2^(m_k - M) acc_k / (2^(sink*log2e - M) + sum_k 2^(m_k - M) l_k)
// m_k, l_k, acc_k are the log2-domain running max, denominator and
// unnormalised output of piece k (without the sink).
//
// One warp per (split token, head): lane k loads (m_k, l_k) of piece k, the
// maxima and denominator are warp reductions, then every lane accumulates
// 16 values of D (D = 512; 4 x 16-byte loads per piece, independent across
// pieces) and stores them as bf16.  Warps past the actual number of split
// tokens exit at once (the grid is sized for the worst case so that it can
// be captured in a CUDA graph).
constexpr int kCombineWarps = 8;

template <int D>
__global__ void __launch_bounds__(kCombineWarps * 32)
combine_kernel(const float* __restrict__ attn_sink, int H, __nv_bfloat16* __restrict__ out,
               const WsHeader* __restrict__ hdr, const int4* __restrict__ splits,
               const float2* __restrict__ part_ml, const float* __restrict__ part_o) {
  // lane l owns the 4-value groups at d = 4l + 128g (16 values for D = 512;
  // for D = 64 only lanes 0..15 hold a group)
  constexpr int kGroups = D >= 128 ? D / 128 : 1;
  constexpr int kPer = 4 * kGroups;
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int item = blockIdx.x * kCombineWarps + (threadIdx.x >> 5);
  if (item >= hdr->n_split * H) return;
  const int si = item / H, h = item % H;
  const int4 sp = splits[si];
  const int t = sp.x, row0 = sp.y, np = sp.z;
  const float ms = attn_sink[h] * kLog2e;
  // maxima and denominator over the pieces (lanes stride over them)
  float mk = -INFINITY;
  for (int k = lane; k < np; k += 32) mk = fmaxf(mk, part_ml[(size_t)(row0 + k) * H + h].x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mk = fmaxf(mk, __shfl_xor_sync(0xffffffffu, mk, o));
  const float M = fmaxf(ms, mk);
  const bool dead = (ms == INFINITY) || (M == -INFINITY);
  float den = 0.f;
  for (int k = lane; k < np; k += 32) {
    const float2 ml = part_ml[(size_t)(row0 + k) * H + h];
    den += dead ? 0.f : ml.y * ex2_approx(ml.x - M);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
  den += dead ? 1.f : ex2_approx(ms - M);
  float acc[kPer];
#pragma unroll
  for (int e = 0; e < kPer; ++e) acc[e] = 0.f;
  if (!dead) {
    const int d0 = lane * 4;  // this lane's 4-value groups at d0 + 128*j
    for (int k0 = 0; k0 < np; k0 += 32) {
      // weight of piece k0 + j lives in lane j
      const int kk = k0 + lane;
      const float wl = kk < np ? ex2_approx(part_ml[(size_t)(row0 + kk) * H + h].x - M) : 0.f;
      const int nk = min(32, np - k0);
#pragma unroll 4
      for (int j = 0; j < nk; ++j) {
        const float wk = __shfl_sync(0xffffffffu, wl, j);
        const float* o = part_o + ((size_t)(row0 + k0 + j) * H + h) * D + d0;
#pragma unroll
        for (int g = 0; g < kGroups; ++g) {
          if (D < 128 && d0 >= D) break;
          const float4 v = *reinterpret_cast<const float4*>(o + 128 * g);
          acc[4 * g + 0] += wk * v.x;
          acc[4 * g + 1] += wk * v.y;
          acc[4 * g + 2] += wk * v.z;
          acc[4 * g + 3] += wk * v.w;
        }
      }
    }
  }
  const float inv = dead ? 0.f : 1.f / den;
  __nv_bfloat16* orow = out + ((size_t)t * H + h) * D + lane * 4;
#pragma unroll
  for (int g = 0; g < kGroups; ++g) {
    if (D < 128 && lane * 4 >= D) break;
    // "+ 0.f" turns -0 into +0 (a factor of 0 when the sink is +inf)
    __nv_bfloat162 a = __floats2bfloat162_rn(acc[4 * g] * inv + 0.f, acc[4 * g + 1] * inv + 0.f);
    __nv_bfloat162 b = __floats2bfloat162_rn(acc[4 * g + 2] * inv + 0.f, acc[4 * g + 3] * inv + 0.f);
    uint2 pk;
    pk.x = *reinterpret_cast<uint32_t*>(&a);
    pk.y = *reinterpret_cast<uint32_t*>(&b);
    *reinterpret_cast<uint2*>(orow + 128 * g) = pk;
  }
}

}  // namespace

cudaError_t launch_plan(const int32_t* kv_indptr, int N, int64_t total_indices,
                        const LaunchPlan& lp, void* ws, const WsLayout& L, cudaStream_t st) {
  char* base = static_cast<char*>(ws);
  return launch_pdl(plan_kernel, dim3(1), dim3(kPlanThreads), 0, st, kv_indptr, N,
                    (long long)total_indices, lp.hg, lp.grid, lp.tile, lp.min_chunk,
                    reinterpret_cast<WsHeader*>(base),
                    reinterpret_cast<int4*>(base + L.units_off),
                    reinterpret_cast<int4*>(base + L.split_off));
}

cudaError_t launch_scan_plan(int N, int64_t capacity, int32_t* kv_indptr, int32_t* status,
                             const LaunchPlan& lp, void* ws, const WsLayout& L, cudaStream_t st) {
  char* base = static_cast<char*>(ws);
  return launch_pdl(scan_plan_kernel, dim3(1), dim3(kPlanThreads), 0, st, N, capacity, kv_indptr,
                    status, lp.hg, lp.grid, lp.tile, lp.min_chunk,
                    reinterpret_cast<WsHeader*>(base),
                    reinterpret_cast<int4*>(base + L.units_off),
                    reinterpret_cast<int4*>(base + L.split_off));
}

cudaError_t launch_combine(const float* attn_sink, int N, int H, int D, void* out, void* ws,
                           const WsLayout& L, int num_sms, cudaStream_t st) {
  (void)N;
  (void)num_sms;
  if (L.s_max == 0) return cudaSuccess;
  char* base = static_cast<char*>(ws);
  const long long items = (long long)L.s_max * H;
  const int blocks = (int)((items + kCombineWarps - 1) / kCombineWarps);
  auto args = [&](auto kernel) {
    return launch_pdl(kernel, dim3(blocks), dim3(kCombineWarps * 32), 0, st, attn_sink, H,
                      static_cast<__nv_bfloat16*>(out), reinterpret_cast<const WsHeader*>(base),
                      reinterpret_cast<const int4*>(base + L.split_off),
                      reinterpret_cast<const float2*>(base + L.ml_off),
                      reinterpret_cast<const float*>(base + L.o_off));
  };
  switch (D) {
    case 64: return args(combine_kernel<64>);
    case 128: return args(combine_kernel<128>);
    case 256: return args(combine_kernel<256>);
    case 512: return args(combine_kernel<512>);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace sda
