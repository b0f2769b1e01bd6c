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
#include "sda_scatter.cuh"

namespace sda {

namespace {

constexpr int kPlanThreads = 1024;
static_assert(kMaxPlanGrid <= kPlanThreads, "one plan thread per CTA of the grid");

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

// First index i in [lo, hi) with a[i] > x (hi if none); a non-decreasing.
__device__ __forceinline__ int upper_index(const int* a, int lo, int hi, int x) {
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (a[mid] > x) hi = mid;
    else lo = mid + 1;
  }
  return lo;
}
// First index i in [lo, hi) with a[i] >= x (hi if none); a non-decreasing.
__device__ __forceinline__ int lower_index(const int* a, int lo, int hi, int x) {
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (a[mid] >= x) hi = mid;
    else lo = mid + 1;
  }
  return lo;
}

// The work plan: each head group's sequence of KV tiles (the non-empty
// tokens in token order, ceil(L_t / tile) tiles each) is cut into at most
// grid / hg contiguous ranges of nearly equal tile counts, one per CTA.  The
// number of ranges Ga is the smallest that reaches the least possible
// maximum, Wmin = ceil(T / (grid / hg)) tiles; a range boundary that falls
// within Wmin / 16 tiles of a token boundary moves onto it, so that a token
// is cut only where that buys balance.  A token cut by k boundaries becomes
// k + 1 pieces (units with partial rows, merged by the combine kernel).
// CTA g * (grid / hg) + r takes range r of head group g, so the CTAs that
// read a token's rows for different head groups run in step and share them
// through L2.  Zero-length tokens (out = 0) are dealt round-robin over all
// CTAs, ahead of each CTA's range.
//
// Outputs: cta_start[b] .. cta_start[b + 1] is CTA b's contiguous run of
// the unit list; the split list holds (token, first partial row, pieces).
// Scratch: ctok[j] = j-th non-empty token (zero-length tokens from the back),
// ctp[j] = tiles before it (ctp[NNZ] = T).
__device__ __forceinline__ void plan_body(const int32_t* __restrict__ indptr, int N,
                                          long long total_indices, int hg, int grid, int tile,
                                          WsHeader* __restrict__ hdr, int4* __restrict__ units,
                                          int4* __restrict__ splits, int* __restrict__ cta_start,
                                          int* __restrict__ ctok, int* __restrict__ ctp,
                                          bool check_indptr) {
  __shared__ int warp_sums[32];
  __shared__ int s_total[2];
  __shared__ int sB[kMaxPlanGrid + 1];      // range boundaries (tiles)
  __shared__ int s_lo[kMaxPlanGrid];        // first non-empty token of range r
  __shared__ int s_start[kMaxPlanGrid + 1]; // start of CTA b's unit run
  __shared__ int s_nz[kMaxPlanGrid];        // zero-length units of CTA b

  // kv_indptr must be a true prefix sum inside [0, total_indices]; otherwise
  // nothing is planned (out is left unwritten) and the error word reads 2, so
  // that no kernel ever reads kv_indices out of bounds.  (A prefix sum that
  // the builder's scan wrote is one by construction.)
  int bad = 0;
  for (int t = threadIdx.x; check_indptr && t <= N; t += kPlanThreads) {
    const int v = indptr[t];
    if (v < 0 || (long long)v > total_indices || (t < N && indptr[t + 1] < v)) bad = 1;
  }
  if (__syncthreads_or(bad)) {
    for (int b = threadIdx.x; b <= grid; b += kPlanThreads) cta_start[b] = 0;
    if (threadIdx.x == 0) {
      hdr->n_units = 0;
      hdr->n_split = 0;
      hdr->n_parts = 0;
      hdr->chunk = 0;
      hdr->error = 2;
    }
    return;
  }

  // pass 1: compact the non-empty tokens and scan their tile counts
  int nnz = 0, T = 0;
  for (int t0 = 0; t0 < N; t0 += kPlanThreads) {
    const int t = t0 + threadIdx.x;
    const int L = t < N ? indptr[t + 1] - indptr[t] : 0;
    const int nz = L > 0 ? 1 : 0;
    const int nt = (L + tile - 1) / tile;
    const int rank = block_exclusive_scan(nz, warp_sums, &s_total[0]) + nnz;
    const int tp = block_exclusive_scan(nt, warp_sums, &s_total[1]) + T;
    if (t < N) {
      if (nz) {
        ctok[rank] = t;
        ctp[rank] = tp;
      } else {
        ctok[N - 1 - (t - rank)] = t;  // zero-length token number t - rank
      }
    }
    nnz += s_total[0];
    T += s_total[1];
    __syncthreads();  // s_total is rewritten by the next chunk
  }
  if (threadIdx.x == 0) ctp[nnz] = T;
  __syncthreads();  // ctok / ctp visible to the whole CTA
  const int NZ = N - nnz;
  const int Gh = grid / hg;
  const int Wmin = T > 0 ? (T + Gh - 1) / Gh : 0;
  const int Ga = T > 0 ? (T + Wmin - 1) / Wmin : 0;  // ranges in use per head group (<= Gh)
  const int snap = Wmin / 16;

  // range boundaries: nominal r*T/Ga, moved onto a token boundary within
  // snap tiles (nominal boundaries are >= Wmin/2 apart and move by at most
  // Wmin/16, so they stay strictly increasing: no range is empty)
  for (int r = threadIdx.x; r <= Ga; r += kPlanThreads) {
    int x = Ga > 0 ? (int)(((long long)r * T) / Ga) : 0;
    if (r > 0 && r < Ga) {
      const int a = upper_index(ctp, 0, nnz + 1, x) - 1;  // ctp[a] <= x < ctp[a + 1]
      const int dl = x - ctp[a], dh = ctp[a + 1] - x;
      if (dl <= dh && dl <= snap) x = ctp[a];
      else if (dh < dl && dh <= snap) x = ctp[a + 1];
    }
    sB[r] = x;
  }
  __syncthreads();

  // units per CTA: its share of the zero-length (token, head group) pairs,
  // then one per token its range touches
  const int zp_total = hg * NZ;
  {
    const int b = threadIdx.x;  // grid <= kMaxPlanGrid <= kPlanThreads
    int total = 0;
    if (b < grid) {
      const int nzb = b < zp_total ? (zp_total - 1 - b) / grid + 1 : 0;
      const int g = b / Gh, r = b % Gh;
      int cnt = 0;
      if (g < hg && r < Ga) {
        const int lo = upper_index(ctp, 1, nnz + 1, sB[r]) - 1;  // first j with ctp[j+1] > B[r]
        const int hi = lower_index(ctp, 0, nnz, sB[r + 1]) - 1;  // last j with ctp[j] < B[r+1]
        cnt = hi - lo + 1;
        if (g == 0) s_lo[r] = lo;
      }
      s_nz[b] = nzb;
      total = nzb + cnt;
    }
    const int start = block_exclusive_scan(total, warp_sums, &s_total[0]);
    if (b < grid) {
      s_start[b] = start;
      cta_start[b] = start;
    }
    if (b == 0) {
      s_start[grid] = s_total[0];
      cta_start[grid] = s_total[0];
    }
  }
  __syncthreads();

  // pass 2: the units of every non-empty token and the split list
  int part_carry = 0, split_carry = 0;
  for (int j0 = 0; j0 < nnz; j0 += kPlanThreads) {
    const int j = j0 + threadIdx.x;
    int f = 0, l = -1, a0 = 0, a1 = 0;
    if (j < nnz) {
      a0 = ctp[j];
      a1 = ctp[j + 1];
      f = upper_index(sB, 0, Ga + 1, a0) - 1;      // range holding the token's first tile
      l = upper_index(sB, 0, Ga + 1, a1 - 1) - 1;  // and its last
    }
    const int pieces = l - f + 1;
    const bool split = pieces > 1;
    const int part_base = block_exclusive_scan(split ? pieces : 0, warp_sums, &s_total[0]) + part_carry;
    const int split_idx = block_exclusive_scan(split ? 1 : 0, warp_sums, &s_total[1]) + split_carry;
    if (j < nnz) {
      const int t = ctok[j];
      const int begin0 = indptr[t], L = indptr[t + 1] - begin0;
      if (split) splits[split_idx] = make_int4(t, part_base, pieces, 0);
      for (int r = f; r <= l; ++r) {
        const int lo_t = max(a0, sB[r]) - a0, hi_t = min(a1, sB[r + 1]) - a0;  // tiles of the token
        const int begin = begin0 + lo_t * tile;
        const int len = min(L, hi_t * tile) - lo_t * tile;
        const int row = split ? part_base + (r - f) : -1;
        for (int g = 0; g < hg; ++g) {
          const int b = g * Gh + r;
          units[s_start[b] + s_nz[b] + (j - s_lo[r])] = make_int4(t, begin, len, make_unit_meta(g, row));
        }
      }
    }
    part_carry += s_total[0];
    split_carry += s_total[1];
    __syncthreads();
  }
  // zero-length (token, head group) pairs, round-robin over the CTAs
  for (int zp = threadIdx.x; zp < zp_total; zp += kPlanThreads) {
    const int g = zp / NZ, z = zp % NZ;
    const int t = ctok[N - 1 - z];
    const int b = zp % grid, k = zp / grid;
    units[s_start[b] + k] = make_int4(t, indptr[t], 0, make_unit_meta(g, -1));
  }
  if (threadIdx.x == 0) {
    hdr->n_units = s_start[grid];
    hdr->n_split = split_carry;
    hdr->n_parts = part_carry;
    hdr->chunk = Wmin * tile;
    hdr->error = 0;
  }
}

// Batches of up to kPlanSmemTokens tokens keep the plan's token arrays (ctok,
// ctp) in the CTA's shared memory: the boundary and token passes run binary
// searches over them, and a search through global memory would pay a
// dependent round trip per step.  Larger batches use the workspace copies.
constexpr int kPlanSmemTokens = 12288;
__host__ __device__ constexpr size_t plan_dyn_smem(int N) {
  return N <= kPlanSmemTokens ? (size_t)(2 * (N > 0 ? N : 1) + 1) * 4 : 0;
}
__device__ __forceinline__ void plan_token_arrays(int N, int*& ctok, int*& ctp) {
  extern __shared__ int plan_dyn[];
  if (N <= kPlanSmemTokens) {
    ctok = plan_dyn;
    ctp = plan_dyn + (N > 0 ? N : 1);
  }
}

__global__ void __launch_bounds__(kPlanThreads)
plan_kernel(const int32_t* __restrict__ indptr, int N, long long total_indices, int hg, int grid,
            int tile, WsHeader* __restrict__ hdr, int4* __restrict__ units,
            int4* __restrict__ splits, int* __restrict__ cta_start, int* ctok, int* ctp) {
  pdl_wait();
  pdl_trigger();
  plan_token_arrays(N, ctok, ctp);
  plan_body(indptr, N, total_indices, hg, grid, tile, hdr, units, splits, cta_start, ctok, ctp, true);
}

// The work plan beside the index builder's scatter (sda_build_decode): both
// need only the scanned kv_indptr, so CTA 0 plans while the other CTAs
// scatter (one-token CTAs, or FLAT over the packed output).
template <bool FLAT>
__global__ void __launch_bounds__(kPlanThreads)
scatter_plan_kernel(ScatterArgs sa, long long capacity, int hg, int grid, int tile,
                    WsHeader* __restrict__ hdr, int4* __restrict__ units, int4* __restrict__ splits,
                    int* __restrict__ cta_start, int* ctok, int* ctp) {
  pdl_wait();
  pdl_trigger();
  if (blockIdx.x == 0) {
    plan_token_arrays(sa.N, ctok, ctp);
    plan_body(sa.kv_indptr, sa.N, capacity, hg, grid, tile, hdr, units, splits, cta_start, ctok, ctp,
              false);
  } else if (FLAT) {
    extern __shared__ int32_t scatter_dyn[];
    scatter_flat_body(sa, blockIdx.x - 1, gridDim.x - 1, scatter_dyn);
  } else {
    scatter_tok_body(sa, blockIdx.x - 1, gridDim.x - 1);
  }
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
// pieces) and stores them as bf16.  The split entry is read together with
// the header, and the first two pieces' values together with the (m, l)
// pairs, so a warp waits on two memory round trips.  Warps past the actual number of split
// tokens exit at once (the grid is sized for the worst case so that it can
// be captured in a CUDA graph).
constexpr int kCombineWarps = 8;

template <int D>
__global__ void __launch_bounds__(kCombineWarps * 32)
combine_kernel(const float* __restrict__ attn_sink, int H, __nv_bfloat16* __restrict__ out,
               const WsHeader* __restrict__ hdr, const int4* __restrict__ splits, int s_cap,
               const float2* __restrict__ part_ml, const float* __restrict__ part_o) {
  // lane l owns the 4-value groups at d = 4l + 128g (16 values for D = 512;
  // for D = 64 only lanes 0..15 hold a group)
  constexpr int kGroups = D >= 128 ? D / 128 : 1;
  constexpr int kPer = 4 * kGroups;
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int item = blockIdx.x * kCombineWarps + (threadIdx.x >> 5);
  const int si = item / H, h = item % H;
  const int n_split = hdr->n_split;
  const int4 sp = splits[si < s_cap ? si : 0];  // read together with the header
  if (item >= n_split * H) return;
  const int t = sp.x, row0 = sp.y, np = sp.z;  // np >= 2
  const float ms = attn_sink[h] * kLog2e;
  const int d0 = lane * 4;  // this lane's 4-value groups at d0 + 128*g
  const bool holds = D >= 128 || d0 < D;
  // the pieces' (m, l) (lane k: piece k) and the first two pieces' partial
  // outputs, all in flight together
  const float2 ml0 = lane < np ? part_ml[(size_t)(row0 + lane) * H + h] : make_float2(-INFINITY, 0.f);
  float4 v0[kGroups], v1[kGroups];
  {
    const float* o0 = part_o + ((size_t)row0 * H + h) * D + d0;
    const float* o1 = part_o + ((size_t)(row0 + 1) * H + h) * D + d0;
#pragma unroll
    for (int g = 0; g < kGroups; ++g) {
      v0[g] = holds ? *reinterpret_cast<const float4*>(o0 + 128 * g) : make_float4(0.f, 0.f, 0.f, 0.f);
      v1[g] = holds ? *reinterpret_cast<const float4*>(o1 + 128 * g) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  // maxima and denominator over the pieces (lanes stride over them)
  float mk = ml0.x;
  for (int k = lane + 32; k < np; k += 32) mk = fmaxf(mk, part_ml[(size_t)(row0 + k) * H + h].x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mk = fmaxf(mk, __shfl_xor_sync(0xffffffffu, mk, o));
  const float M = fmaxf(ms, mk);
  const bool dead = (ms == INFINITY) || (M == -INFINITY);
  float den = (dead || lane >= np) ? 0.f : ml0.y * ex2_approx(ml0.x - M);
  for (int k = lane + 32; k < np; k += 32) {
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
    for (int k0 = 0; k0 < np; k0 += 32) {
      // weight of piece k0 + j lives in lane j
      const int kk = k0 + lane;
      const float wl = kk < np ? ex2_approx((k0 == 0 ? ml0.x : part_ml[(size_t)(row0 + kk) * H + h].x) - M) : 0.f;
      const int nk = min(32, np - k0);
      int j = 0;
      if (k0 == 0) {  // the two pieces already loaded
#pragma unroll
        for (int p2 = 0; p2 < 2; ++p2) {
          const float wk = __shfl_sync(0xffffffffu, wl, p2);
#pragma unroll
          for (int g = 0; g < kGroups; ++g) {
            const float4 v = p2 ? v1[g] : v0[g];
            acc[4 * g + 0] += wk * v.x;
            acc[4 * g + 1] += wk * v.y;
            acc[4 * g + 2] += wk * v.z;
            acc[4 * g + 3] += wk * v.w;
          }
        }
        j = 2;
      }
#pragma unroll 4
      for (; j < nk; ++j) {
        const float wk = __shfl_sync(0xffffffffu, wl, j);
        const float* o = part_o + ((size_t)(row0 + k0 + j) * H + h) * D + d0;
#pragma unroll
        for (int g = 0; g < kGroups; ++g) {
          if (!holds) break;
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
  static const cudaError_t attr = cudaFuncSetAttribute(
      plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)plan_dyn_smem(kPlanSmemTokens));
  if (attr != cudaSuccess) return attr;
  return launch_pdl(plan_kernel, dim3(1), dim3(kPlanThreads), plan_dyn_smem(N), st, kv_indptr, N,
                    (long long)total_indices, lp.hg, lp.grid, lp.tile,
                    reinterpret_cast<WsHeader*>(base),
                    reinterpret_cast<int4*>(base + L.units_off),
                    reinterpret_cast<int4*>(base + L.split_off),
                    reinterpret_cast<int*>(base + L.cta_off), reinterpret_cast<int*>(base + L.ctok_off),
                    reinterpret_cast<int*>(base + L.ctp_off));
}

cudaError_t launch_scatter_plan(const ScatterArgs& sa, int64_t capacity, const LaunchPlan& lp,
                               void* ws, const WsLayout& L, int num_sms, cudaStream_t st) {
  char* base = static_cast<char*>(ws);
  const ScatterShape sh = scatter_shape(sa.N, capacity, num_sms, kPlanThreads);
  const size_t pd = plan_dyn_smem(sa.N);
  const size_t smem = pd > sh.smem ? pd : sh.smem;
  auto go = [&](auto kernel, int ctas) {
    return launch_pdl(kernel, dim3(1 + ctas), dim3(kPlanThreads), smem, st, sa, (long long)capacity,
                      lp.hg, lp.grid, lp.tile, reinterpret_cast<WsHeader*>(base),
                      reinterpret_cast<int4*>(base + L.units_off),
                      reinterpret_cast<int4*>(base + L.split_off),
                      reinterpret_cast<int*>(base + L.cta_off),
                      reinterpret_cast<int*>(base + L.ctok_off),
                      reinterpret_cast<int*>(base + L.ctp_off));
  };
  static const cudaError_t attr = [] {
    const int most = (int)plan_dyn_smem(kPlanSmemTokens);
    cudaError_t e = cudaFuncSetAttribute(scatter_plan_kernel<true>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, most);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(scatter_plan_kernel<false>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, most);
    return e;
  }();
  if (attr != cudaSuccess) return attr;
  // no lists to write (capacity 0): CTA 0 alone
  if (capacity <= 0) return go(scatter_plan_kernel<false>, 0);
  return sh.flat ? go(scatter_plan_kernel<true>, sh.ctas) : go(scatter_plan_kernel<false>, sh.ctas);
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
                      reinterpret_cast<const int4*>(base + L.split_off), L.s_max,
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
