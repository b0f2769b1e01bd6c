// sda_build.cu -- the decode index builder and the index validator.
//
// The builder packs, per token, its SWA ring slots (state_slot * win + ring)
// and its compressed-cache slots (swa_pages + block_id * K_PER_BLOCK +
// slot_in_block) into the ragged kv_indices / kv_indptr pair the decode
// kernel reads (paged_decode.py docstring, caller convention for unified_kv
// and kv_indices: ragged-packed, no sentinels, padded tokens get an empty
// slice).  Three launches: per-token validation + length, one-CTA scan,
// scatter over the packed output.  Bad descriptors never reach the decode kernel: the
// token's slice is emptied and a status bit is raised (a divide-by-zero in a
// slot translation that produced out-of-range slots and a GPU fault is the
// failure the sglang PR 25898 summary page describes; here win and
// k_per_block are checked on the host and every emitted slot is in range).
#include "sda_internal.cuh"
#include "sda_scan.cuh"

namespace sda {

namespace {

// Length pass, in two independent parts that share one launch of a single
// wave of CTAs:
//  * tokens (grid-stride, one thread each): every per-token field is
//    checked, and kv_indptr[t + 1] receives the token's length, or
//    -(status bits) for a bad token -- assuming its compressed entries are
//    good;
//  * compressed entries: CTA b checks an equal slice of the entry array,
//    four entries per 16-byte load, and writes flags[b] != 0 if the slice
//    holds a bad entry.  Every token's list, however long, is spread over
//    the whole grid this way.
// The scan re-checks the tokens whose entries overlap a flagged slice (see
// EntryCheck), so the lists and status bits are exactly those of checking
// every token's entries with the token.
constexpr int kLenThreads = 256;
constexpr int kLenCtasPerSm = 4;
constexpr int kLenUnroll = 2;

__global__ void __launch_bounds__(kLenThreads, kLenCtasPerSm)
build_len_kernel(const int32_t* __restrict__ state_slot, const int32_t* __restrict__ swa_len,
                 const int32_t* __restrict__ swa_head, const int32_t* __restrict__ comp_indptr,
                 const int32_t* __restrict__ comp_block, const int32_t* __restrict__ comp_slot,
                 int64_t comp_total, int N, int win, int k_per_block, int64_t swa_pages,
                 int64_t total_pages, int64_t chunks_per_cta, int32_t* __restrict__ kv_indptr,
                 int32_t* __restrict__ flags) {
  pdl_wait();
  pdl_trigger();
  // this CTA's slice of the entries: chunks [qa, qe) of 4 entries
  const int64_t nq = (comp_total + 3) >> 2;
  const int64_t qa = (int64_t)blockIdx.x * chunks_per_cta;
  const int64_t qe = qa + chunks_per_cta < nq ? qa + chunks_per_cta : nq;
  const bool vec =
      ((reinterpret_cast<uintptr_t>(comp_block) | reinterpret_cast<uintptr_t>(comp_slot)) & 15) == 0;
  const int4* cb4 = reinterpret_cast<const int4*>(comp_block);
  const int4* cs4 = reinterpret_cast<const int4*>(comp_slot);
  int32_t bad = 0;
  for (int64_t qb = qa + threadIdx.x; qb < qe; qb += (int64_t)kLenUnroll * kLenThreads) {
    int4 B[kLenUnroll], S[kLenUnroll];
#pragma unroll
    for (int u = 0; u < kLenUnroll; ++u) {
      const int64_t q = qb + (int64_t)u * kLenThreads;
      if (vec && q < qe && 4 * q + 4 <= comp_total) {
        B[u] = __ldg(cb4 + q);
        S[u] = __ldg(cs4 + q);
      }
    }
#pragma unroll
    for (int u = 0; u < kLenUnroll; ++u) {
      const int64_t q = qb + (int64_t)u * kLenThreads;
      if (q >= qe) break;
      if (vec && 4 * q + 4 <= comp_total) {
        bad |= entry_bad(B[u].x, S[u].x, k_per_block, swa_pages, total_pages) |
               entry_bad(B[u].y, S[u].y, k_per_block, swa_pages, total_pages) |
               entry_bad(B[u].z, S[u].z, k_per_block, swa_pages, total_pages) |
               entry_bad(B[u].w, S[u].w, k_per_block, swa_pages, total_pages);
      } else {  // unaligned arrays, or the chunk that runs past their end
        for (int64_t e = 4 * q; e < 4 * q + 4 && e < comp_total; ++e)
          bad |= entry_bad(comp_block[e], comp_slot[e], k_per_block, swa_pages, total_pages);
      }
    }
  }
  // the tokens' own fields and lengths
  for (int t = blockIdx.x * kLenThreads + threadIdx.x; t < N; t += gridDim.x * kLenThreads) {
    const int32_t ss = state_slot[t], n_swa = swa_len[t], head = swa_head[t];
    const int32_t c0 = comp_indptr[t], c1 = comp_indptr[t + 1];
    int32_t tb = 0;
    int64_t len = 0;
    if (ss >= 0) {
      if (n_swa < 0 || n_swa > win) tb |= 1;
      else if (n_swa > 0 && (head < 0 || head >= win)) tb |= 2;
      else if (n_swa > 0 && (int64_t)ss * win + win > swa_pages) tb |= 16;
      if (c0 < 0 || c1 < c0 || (int64_t)c1 > comp_total) tb |= 4;
      len = (int64_t)(n_swa > 0 ? n_swa : 0) + (c1 > c0 ? c1 - c0 : 0);
    }
    kv_indptr[t + 1] = tb ? -tb : (int32_t)(len > 0x7fffffff ? 0x7fffffff : len);
  }
  const int b8 = __syncthreads_or(bad & 8), b16 = __syncthreads_or(bad & 16);
  if (threadIdx.x == 0) flags[blockIdx.x] = (b8 ? 8 : 0) | (b16 ? 16 : 0);
}

__global__ void __launch_bounds__(kScanThreads)
build_scan_kernel(int N, int64_t capacity, int32_t* __restrict__ kv_indptr,
                  int32_t* __restrict__ status, EntryCheck ec) {
  pdl_wait();
  pdl_trigger();
  build_scan_body(N, capacity, kv_indptr, status, ec);
}

// Scatter pass for batches that fit one wave of CTAs: one CTA per token
// writes its slots at kv_indices[kv_indptr[t] ...]; the token's fields are
// loaded together with its slice bounds (two dependent round trips before
// the compressed entries).
constexpr int kTokThreads = 1024;

__global__ void __launch_bounds__(kTokThreads)
build_scatter_tok_kernel(const int32_t* __restrict__ state_slot, const int32_t* __restrict__ swa_len,
                         const int32_t* __restrict__ swa_head, const int32_t* __restrict__ comp_indptr,
                         const int32_t* __restrict__ comp_block, const int32_t* __restrict__ comp_slot,
                         int N, int win, int k_per_block, int64_t swa_pages,
                         const int32_t* __restrict__ kv_indptr, int32_t* __restrict__ kv_indices) {
  pdl_wait();
  pdl_trigger();
  for (int t = blockIdx.x; t < N; t += gridDim.x) {
    const int32_t o0 = kv_indptr[t], o1 = kv_indptr[t + 1];
    const int32_t ss = state_slot[t], n_swa = swa_len[t], head = swa_head[t], c0 = comp_indptr[t];
    if (o1 <= o0) continue;  // padded, bad or over capacity (uniform)
    const int32_t ns = n_swa > 0 ? n_swa : 0;
    for (int32_t j = threadIdx.x; j < ns; j += kTokThreads) {
      int32_t ring = (int32_t)(((int64_t)head - n_swa + 1 + j) % win);
      if (ring < 0) ring += win;
      kv_indices[o0 + j] = (int32_t)((int64_t)ss * win + ring);
    }
    const int32_t nc = o1 - o0 - ns;
#pragma unroll 8
    for (int32_t i = threadIdx.x; i < nc; i += kTokThreads)
      kv_indices[o0 + ns + i] =
          (int32_t)(swa_pages + (int64_t)comp_block[c0 + i] * k_per_block + comp_slot[c0 + i]);
  }
}

// Scatter pass for larger batches, flat over the packed output: thread i writes the outputs
// [4i, 4i + 4) (grid-stride), finding the token of the first by a binary
// search in kv_indptr (staged in shared memory for batches of up to
// kScatterSmemTokens tokens) and walking on from there.  Every token's list
// is spread over as many threads as it has outputs / 4, however long it is.
constexpr int kScatterThreads = 256;
constexpr int kScatterPer = 4;
constexpr int kScatterSmemTokens = 8191;

__global__ void __launch_bounds__(kScatterThreads)
build_scatter_kernel(const int32_t* __restrict__ state_slot, const int32_t* __restrict__ swa_len,
                     const int32_t* __restrict__ swa_head, const int32_t* __restrict__ comp_indptr,
                     const int32_t* __restrict__ comp_block, const int32_t* __restrict__ comp_slot,
                     int N, int win, int k_per_block, int64_t swa_pages,
                     const int32_t* __restrict__ kv_indptr, int32_t* __restrict__ kv_indices) {
  extern __shared__ int32_t s_ptr[];
  pdl_wait();
  pdl_trigger();
  const bool staged = N <= kScatterSmemTokens;
  if (staged) {  // (uniform)
    for (int i = threadIdx.x; i <= N; i += kScatterThreads) s_ptr[i] = kv_indptr[i];
    __syncthreads();
  }
  const int32_t* ptr = staged ? s_ptr : kv_indptr;
  const int32_t total = ptr[N];  // 0 when the lists were emptied (over capacity)
  const int64_t first = (int64_t)blockIdx.x * kScatterThreads * kScatterPer;
  if (first >= total) return;  // the whole CTA: uniform
  const int64_t stride = (int64_t)gridDim.x * kScatterThreads * kScatterPer;
  for (int64_t o0 = first + (int64_t)threadIdx.x * kScatterPer; o0 < total; o0 += stride) {
    // token of each output: a binary search for the first (last t with
    // ptr[t] <= o0; ptr is non-decreasing, ptr[0] = 0 <= o0 < ptr[N]), then
    // a walk past the next list ends
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
    // every load of the kScatterPer outputs in flight together
    int32_t ss[kScatterPer], ns[kScatterPer], hd[kScatterPer], c0[kScatterPer];
#pragma unroll
    for (int k = 0; k < kScatterPer; ++k) {
      ss[k] = state_slot[tk[k]];
      ns[k] = swa_len[tk[k]];
      hd[k] = swa_head[tk[k]];
      c0[k] = comp_indptr[tk[k]];
    }
    int32_t cb[kScatterPer], cs[kScatterPer];
#pragma unroll
    for (int k = 0; k < kScatterPer; ++k) {
      const bool comp = o0 + k < total && jk[k] >= ns[k];
      const int32_t e = c0[k] + (jk[k] - (ns[k] > 0 ? ns[k] : 0));
      cb[k] = comp ? comp_block[e] : 0;
      cs[k] = comp ? comp_slot[e] : 0;
    }
#pragma unroll
    for (int k = 0; k < kScatterPer; ++k) {
      const int64_t o = o0 + k;
      if (o >= total) break;
      int32_t v;
      if (jk[k] < ns[k]) {
        int32_t ring = (int32_t)(((int64_t)hd[k] - ns[k] + 1 + jk[k]) % win);
        if (ring < 0) ring += win;
        v = (int32_t)((int64_t)ss[k] * win + ring);
      } else {
        v = (int32_t)(swa_pages + (int64_t)cb[k] * k_per_block + cs[k]);
      }
      kv_indices[o] = v;
    }
  }
}

__global__ void validate_kernel(const int32_t* __restrict__ kv_indices, int64_t total_indices,
                                const int32_t* __restrict__ kv_indptr, int N,
                                int64_t total_pages, int32_t* __restrict__ status) {
  int32_t flags = 0;
  int32_t n_bad = 0;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (int64_t t = tid; t <= N; t += stride) {
    const int32_t p = kv_indptr[t];
    if (p < 0 || (int64_t)p > total_indices) flags |= 2;
    if (t < N && kv_indptr[t + 1] < p) flags |= 1;
  }
  for (int64_t e = tid; e < total_indices; e += stride) {
    const int32_t s = kv_indices[e];
    if (s < 0 || (int64_t)s >= total_pages) ++n_bad;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    flags |= __shfl_xor_sync(0xffffffffu, flags, o);
    n_bad += __shfl_xor_sync(0xffffffffu, n_bad, o);
  }
  if ((threadIdx.x & 31) == 0) {
    if (n_bad) flags |= 4;
    if (flags) atomicOr(&status[0], flags);
    if (n_bad) atomicAdd(&status[1], n_bad);
  }
}

}  // namespace

EntryCheck entry_check_layout(const int32_t* state_slot, const int32_t* comp_indptr,
                              const int32_t* comp_block, const int32_t* comp_slot,
                              int64_t comp_total, int N, int k_per_block, int64_t swa_pages,
                              int64_t total_pages, int64_t capacity, int32_t* kv_indices,
                              int32_t* status, int num_sms) {
  EntryCheck ec{};
  ec.state_slot = state_slot;
  ec.comp_indptr = comp_indptr;
  ec.comp_block = comp_block;
  ec.comp_slot = comp_slot;
  ec.comp_total = comp_total;
  ec.k_per_block = k_per_block;
  ec.swa_pages = swa_pages;
  ec.total_pages = total_pages;
  // one wave of CTAs, no more than the work needs (a token or kLenUnroll
  // chunks per thread), and no more than kv_indices has room for flags
  // (the scatter overwrites them after the scan has read them); a builder
  // without room keeps its one flag in the status word, which the scan
  // writes last
  const long long nq = (comp_total + 3) / 4;
  const long long per_cta = (long long)kLenThreads * kLenUnroll;
  long long g = (nq + per_cta - 1) / per_cta;
  const long long gt = ((long long)N + kLenThreads - 1) / kLenThreads;
  if (gt > g) g = gt;
  const long long wave = (long long)num_sms * kLenCtasPerSm;
  if (g > wave) g = wave;
  if (g > capacity) g = capacity;
  if (g < 1) g = 1;
  ec.n_flags = (int)g;
  ec.flags = capacity >= g ? kv_indices : status;
  ec.chunks_per_cta = nq > 0 ? (nq + g - 1) / g : 1;
  return ec;
}

cudaError_t launch_build_len(const int32_t* swa_len, const int32_t* swa_head, int N, int win,
                             int32_t* kv_indptr, const EntryCheck& ec, cudaStream_t st) {
  if (N <= 0) return cudaSuccess;
  return launch_pdl(build_len_kernel, dim3(ec.n_flags), dim3(kLenThreads), 0, st, ec.state_slot,
                    swa_len, swa_head, ec.comp_indptr, ec.comp_block, ec.comp_slot, ec.comp_total,
                    N, win, ec.k_per_block, ec.swa_pages, ec.total_pages, ec.chunks_per_cta,
                    kv_indptr, const_cast<int32_t*>(ec.flags));
}

cudaError_t launch_build_scatter(const int32_t* state_slot, const int32_t* swa_len,
                                 const int32_t* swa_head, const int32_t* comp_indptr,
                                 const int32_t* comp_block, const int32_t* comp_slot, int N,
                                 int win, int k_per_block, int64_t swa_pages, int64_t capacity,
                                 const int32_t* kv_indptr, int32_t* kv_indices, cudaStream_t st) {
  if (N <= 0 || capacity <= 0) return cudaSuccess;
  DeviceCaps caps;
  const cudaError_t ce = device_caps(&caps);
  if (ce != cudaSuccess) return ce;
  if (N <= 2 * caps.num_sms)  // one wave of one-token CTAs
    return launch_pdl(build_scatter_tok_kernel, dim3(N), dim3(kTokThreads), 0, st, state_slot,
                      swa_len, swa_head, comp_indptr, comp_block, comp_slot, N, win, k_per_block,
                      swa_pages, kv_indptr, kv_indices);
  // enough threads for the capacity, at most one wave (grid-stride beyond)
  const long long per_cta = (long long)kScatterThreads * kScatterPer;
  const long long need = (capacity + per_cta - 1) / per_cta;
  const long long wave = (long long)caps.num_sms * (2048 / kScatterThreads);
  const int blocks = (int)(need < wave ? need : wave);
  const size_t smem = N <= kScatterSmemTokens ? (size_t)(N + 1) * sizeof(int32_t) : 0;
  return launch_pdl(build_scatter_kernel, dim3(blocks), dim3(kScatterThreads), smem, st, state_slot,
                    swa_len, swa_head, comp_indptr, comp_block, comp_slot, N, win, k_per_block,
                    swa_pages, kv_indptr, kv_indices);
}

cudaError_t launch_build_indices(const int32_t* state_slot, const int32_t* swa_len,
                                 const int32_t* swa_head, const int32_t* comp_indptr,
                                 const int32_t* comp_block, const int32_t* comp_slot,
                                 int64_t comp_total, int N, int win, int k_per_block,
                                 int64_t swa_pages, int64_t total_pages, int32_t* kv_indices,
                                 int64_t capacity, int32_t* kv_indptr, int32_t* status,
                                 cudaStream_t st) {
  DeviceCaps caps;
  cudaError_t e = device_caps(&caps);
  if (e != cudaSuccess) return e;
  const EntryCheck ec = entry_check_layout(state_slot, comp_indptr, comp_block, comp_slot,
                                           comp_total, N, k_per_block, swa_pages, total_pages,
                                           capacity, kv_indices, status, caps.num_sms);
  e = launch_build_len(swa_len, swa_head, N, win, kv_indptr, ec, st);
  if (e == cudaSuccess)
    e = launch_pdl(build_scan_kernel, dim3(1), dim3(kScanThreads), 0, st, N, capacity, kv_indptr,
                   status, ec);
  if (e == cudaSuccess)
    e = launch_build_scatter(state_slot, swa_len, swa_head, comp_indptr, comp_block, comp_slot, N,
                             win, k_per_block, swa_pages, capacity, kv_indptr, kv_indices, st);
  return e;
}

cudaError_t launch_validate(const int32_t* kv_indices, int64_t total_indices,
                            const int32_t* kv_indptr, int N, int64_t total_pages,
                            int32_t* status, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(status, 0, 2 * sizeof(int32_t), st);
  if (e != cudaSuccess) return e;
  const int threads = 256;
  int64_t work = total_indices > (int64_t)N + 1 ? total_indices : (int64_t)N + 1;
  int blocks = (int)((work + threads - 1) / threads);
  if (blocks > 1024) blocks = 1024;
  if (blocks < 1) blocks = 1;
  validate_kernel<<<blocks, threads, 0, st>>>(kv_indices, total_indices, kv_indptr, N,
                                              total_pages, status);
  return cudaGetLastError();
}

}  // namespace sda
