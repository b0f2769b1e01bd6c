// sda_scatter.cuh -- the index builder's scatter (packed slot lists from the
// descriptors and the scanned kv_indptr), shared by its own kernels
// (sda_build.cu) and by the kernel that runs it beside the work plan
// (sda_plan.cu).  Both bodies work for any block size.
#pragma once

#include <cstdint>

#include "sda_internal.cuh"

namespace sda {

struct ScatterArgs {
  const int32_t* state_slot;
  const int32_t* swa_len;
  const int32_t* swa_head;
  const int32_t* comp_indptr;
  const int32_t* comp_block;
  const int32_t* comp_slot;
  int N;
  int win;
  int k_per_block;
  int64_t swa_pages;
  const int32_t* kv_indptr;  // scanned: a non-decreasing prefix sum, kv_indptr[0] = 0
  int32_t* kv_indices;
};

constexpr int kTokThreads = 1024;         // threads of a one-token CTA
constexpr int kScatterPer = 4;            // outputs per thread of the flat scatter
constexpr int kScatterSmemTokens = 8191;  // flat scatter: kv_indptr staged up to this N

// Slot j of a token: its SWA ring slots first (oldest -> newest), then its
// compressed entries in input order.
__device__ __forceinline__ int32_t swa_slot(int32_t ss, int32_t n_swa, int32_t head, int32_t j,
                                            int win) {
  int32_t ring = (int32_t)(((int64_t)head - n_swa + 1 + j) % win);
  if (ring < 0) ring += win;
  return (int32_t)((int64_t)ss * win + ring);
}

// One token per CTA (tokens cta, cta + ncta, ...): the token's fields are
// loaded with its slice bounds, so the compressed entries are the second
// dependent round trip.  For batches that fit one wave of such CTAs.
__device__ __forceinline__ void scatter_tok_body(const ScatterArgs& a, int cta, int ncta) {
  for (int t = cta; t < a.N; t += ncta) {
    const int32_t o0 = a.kv_indptr[t], o1 = a.kv_indptr[t + 1];
    const int32_t ss = a.state_slot[t], n_swa = a.swa_len[t], head = a.swa_head[t];
    const int32_t c0 = a.comp_indptr[t];
    if (o1 <= o0) continue;  // padded, bad or over capacity (uniform)
    const int32_t ns = n_swa > 0 ? n_swa : 0;
    for (int32_t j = threadIdx.x; j < ns; j += blockDim.x)
      a.kv_indices[o0 + j] = swa_slot(ss, n_swa, head, j, a.win);
    const int32_t nc = o1 - o0 - ns;
#pragma unroll 8
    for (int32_t i = threadIdx.x; i < nc; i += blockDim.x)
      a.kv_indices[o0 + ns + i] =
          (int32_t)(a.swa_pages + (int64_t)a.comp_block[c0 + i] * a.k_per_block + a.comp_slot[c0 + i]);
  }
}

// Flat over the packed output: thread i of CTA cta writes the outputs
// [4i, 4i + 4) of the CTA's block of blockDim.x * 4 (grid-stride over ncta
// CTAs), finding the first one's token by a binary search in kv_indptr
// (staged in s_ptr, (N + 1) ints, for N <= kScatterSmemTokens) and the
// others' by a walk; all of a thread's loads are in flight together.  Every
// token's list is spread over as many threads as it has outputs / 4.  Ends
// early (the whole CTA) when the CTA has no outputs.
__device__ __forceinline__ void scatter_flat_body(const ScatterArgs& a, int cta, int ncta,
                                                  int32_t* s_ptr) {
  const int N = a.N;
  const bool staged = N <= kScatterSmemTokens;
  if (staged) {  // (uniform)
    for (int i = threadIdx.x; i <= N; i += blockDim.x) s_ptr[i] = a.kv_indptr[i];
    __syncthreads();
  }
  const int32_t* ptr = staged ? s_ptr : a.kv_indptr;
  const int32_t total = ptr[N];  // 0 when the lists were emptied (over capacity)
  const int64_t per_cta = (int64_t)blockDim.x * kScatterPer;
  const int64_t first = (int64_t)cta * per_cta;
  if (first >= total) return;
  const int64_t stride = (int64_t)ncta * per_cta;
  for (int64_t o0 = first + (int64_t)threadIdx.x * kScatterPer; o0 < total; o0 += stride) {
    // last t with ptr[t] <= o0 (ptr[0] = 0 <= o0 < ptr[N])
    int lo = 0, hi = N - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (ptr[mid] <= o0) lo = mid;
      else hi = mid - 1;
    }
    int tk[kScatterPer];
    int32_t jk[kScatterPer];
    int t = lo;
#pragma unroll
    for (int k = 0; k < kScatterPer; ++k) {
      const int64_t o = o0 + k;
      if (o < total)
        while (o >= ptr[t + 1]) ++t;
      tk[k] = t;
      jk[k] = (int32_t)(o - ptr[t]);
    }
    int32_t ss[kScatterPer], ns[kScatterPer], hd[kScatterPer], c0[kScatterPer];
#pragma unroll
    for (int k = 0; k < kScatterPer; ++k) {
      ss[k] = a.state_slot[tk[k]];
      ns[k] = a.swa_len[tk[k]];
      hd[k] = a.swa_head[tk[k]];
      c0[k] = a.comp_indptr[tk[k]];
    }
    int32_t cb[kScatterPer], cs[kScatterPer];
#pragma unroll
    for (int k = 0; k < kScatterPer; ++k) {
      const bool comp = o0 + k < total && jk[k] >= ns[k];
      const int32_t e = c0[k] + (jk[k] - (ns[k] > 0 ? ns[k] : 0));
      cb[k] = comp ? a.comp_block[e] : 0;
      cs[k] = comp ? a.comp_slot[e] : 0;
    }
#pragma unroll
    for (int k = 0; k < kScatterPer; ++k) {
      const int64_t o = o0 + k;
      if (o >= total) break;
      a.kv_indices[o] = jk[k] < ns[k]
                            ? swa_slot(ss[k], ns[k], hd[k], jk[k], a.win)
                            : (int32_t)(a.swa_pages + (int64_t)cb[k] * a.k_per_block + cs[k]);
    }
  }
}

// The scatter's shape: one-token CTAs while a batch fits one wave of them,
// else the flat body over enough CTAs of `threads` threads for the capacity
// (at most one wave of 2048 threads per SM; grid-stride beyond).
struct ScatterShape {
  bool flat;
  int ctas;
  size_t smem;  // dynamic shared memory of the flat body
};
inline ScatterShape scatter_shape(int N, int64_t capacity, int num_sms, int threads) {
  ScatterShape s{};
  if (N <= 2 * num_sms) {
    s.flat = false;
    s.ctas = N;
    s.smem = 0;
    return s;
  }
  s.flat = true;
  const long long per_cta = (long long)threads * kScatterPer;
  const long long need = (capacity + per_cta - 1) / per_cta;
  const long long wave = (long long)num_sms * (2048 / threads);
  s.ctas = (int)(need < wave ? (need > 0 ? need : 1) : wave);
  s.smem = N <= kScatterSmemTokens ? (size_t)(N + 1) * sizeof(int32_t) : 0;
  return s;
}

}  // namespace sda
