// sda_build.cu -- the decode index builder and the index validator.
//
// The builder packs, per token, its SWA ring slots (state_slot * win + ring)
// and its compressed-cache slots (swa_pages + block_id * K_PER_BLOCK +
// slot_in_block) into the ragged kv_indices / kv_indptr pair the decode
// kernel reads (paged_decode.py docstring, caller convention for unified_kv
// and kv_indices: ragged-packed, no sentinels, padded tokens get an empty
// slice).  Three launches: per-token validation + length, one-CTA scan,
// per-token scatter.  Bad descriptors never reach the decode kernel: the
// token's slice is emptied and a status bit is raised (a divide-by-zero in a
// slot translation that produced out-of-range slots and a GPU fault is the
// failure the sglang PR 25898 summary page describes; here win and
// k_per_block are checked on the host and every emitted slot is in range).
#include "sda_internal.cuh"
#include "sda_scan.cuh"

namespace sda {

namespace {

// One CTA per token in the length and scatter passes; 1024 threads and loops
// unrolled 8 deep keep a long list (e.g. 64 K compressed entries) to a few
// dependent memory round trips.
constexpr int kTokThreads = 1024;

// One CTA per token: check every field, write the length to kv_indptr[t + 1]
// (rewritten in place by the scan), or -(status bits) if the token is bad.
__global__ void __launch_bounds__(kTokThreads)
build_len_kernel(const int32_t* __restrict__ state_slot, const int32_t* __restrict__ swa_len,
                 const int32_t* __restrict__ swa_head, const int32_t* __restrict__ comp_indptr,
                 const int32_t* __restrict__ comp_block, const int32_t* __restrict__ comp_slot,
                 int64_t comp_total, int N, int win, int k_per_block, int64_t swa_pages,
                 int64_t total_pages, int32_t* __restrict__ kv_indptr) {
  pdl_wait();
  pdl_trigger();
  for (int t = blockIdx.x; t < N; t += gridDim.x) {
    int32_t bad = 0;
    int64_t len = 0;
    const int32_t ss = state_slot[t];
    if (ss >= 0) {
      const int32_t n_swa = swa_len[t];
      if (n_swa < 0 || n_swa > win) bad |= 1;
      else if (n_swa > 0 && (swa_head[t] < 0 || swa_head[t] >= win)) bad |= 2;
      else if (n_swa > 0 && (int64_t)ss * win + win > swa_pages) bad |= 16;
      const int32_t c0 = comp_indptr[t], c1 = comp_indptr[t + 1];
      if (c0 < 0 || c1 < c0 || (int64_t)c1 > comp_total) {
        bad |= 4;
      } else {
#pragma unroll 8
        for (int32_t e = c0 + threadIdx.x; e < c1; e += kTokThreads) {
          const int32_t b = comp_block[e], s = comp_slot[e];
          if (b < 0 || s < 0 || s >= k_per_block) bad |= 8;
          else if (swa_pages + (int64_t)b * k_per_block + s >= total_pages) bad |= 16;
        }
      }
      len = (int64_t)(n_swa > 0 ? n_swa : 0) + (c1 > c0 ? c1 - c0 : 0);
    }
    __shared__ int s_bad;  // OR of every thread's findings for token t
    if (threadIdx.x == 0) s_bad = 0;
    __syncthreads();
    if (bad) atomicOr(&s_bad, bad);
    __syncthreads();
    if (threadIdx.x == 0)
      kv_indptr[t + 1] = s_bad ? -s_bad : (int32_t)(len > 0x7fffffff ? 0x7fffffff : len);
    __syncthreads();
  }
}

__global__ void __launch_bounds__(kScanThreads)
build_scan_kernel(int N, int64_t capacity, int32_t* __restrict__ kv_indptr,
                  int32_t* __restrict__ status) {
  pdl_wait();
  pdl_trigger();
  build_scan_body(N, capacity, kv_indptr, status);
}

// One CTA per token: write its slots at kv_indices[kv_indptr[t] ...].
__global__ void __launch_bounds__(kTokThreads)
build_scatter_kernel(const int32_t* __restrict__ state_slot, const int32_t* __restrict__ swa_len,
                     const int32_t* __restrict__ swa_head, const int32_t* __restrict__ comp_indptr,
                     const int32_t* __restrict__ comp_block, const int32_t* __restrict__ comp_slot,
                     int N, int win, int k_per_block, int64_t swa_pages,
                     const int32_t* __restrict__ kv_indptr, int32_t* __restrict__ kv_indices) {
  pdl_wait();
  pdl_trigger();
  for (int t = blockIdx.x; t < N; t += gridDim.x) {
    const int32_t o0 = kv_indptr[t], o1 = kv_indptr[t + 1];
    if (o1 <= o0) continue;  // padded, bad or over capacity
    const int32_t ss = state_slot[t];
    const int32_t n_swa = swa_len[t];
    const int32_t head = swa_head[t];
    for (int32_t j = threadIdx.x; j < n_swa; j += kTokThreads) {
      int32_t ring = (int32_t)(((int64_t)head - n_swa + 1 + j) % win);
      if (ring < 0) ring += win;
      kv_indices[o0 + j] = (int32_t)((int64_t)ss * win + ring);
    }
    const int32_t c0 = comp_indptr[t], c1 = comp_indptr[t + 1];
#pragma unroll 8
    for (int32_t e = c0 + threadIdx.x; e < c1; e += kTokThreads)
      kv_indices[o0 + n_swa + (e - c0)] =
          (int32_t)(swa_pages + (int64_t)comp_block[e] * k_per_block + comp_slot[e]);
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

cudaError_t launch_build_len(const int32_t* state_slot, const int32_t* swa_len,
                             const int32_t* swa_head, const int32_t* comp_indptr,
                             const int32_t* comp_block, const int32_t* comp_slot,
                             int64_t comp_total, int N, int win, int k_per_block,
                             int64_t swa_pages, int64_t total_pages, int32_t* kv_indptr,
                             cudaStream_t st) {
  if (N <= 0) return cudaSuccess;
  const int blocks = N < 65535 ? N : 65535;
  return launch_pdl(build_len_kernel, dim3(blocks), dim3(kTokThreads), 0, st, state_slot, swa_len,
                    swa_head, comp_indptr, comp_block, comp_slot, comp_total, N, win, k_per_block,
                    swa_pages, total_pages, kv_indptr);
}

cudaError_t launch_build_scatter(const int32_t* state_slot, const int32_t* swa_len,
                                 const int32_t* swa_head, const int32_t* comp_indptr,
                                 const int32_t* comp_block, const int32_t* comp_slot, int N,
                                 int win, int k_per_block, int64_t swa_pages,
                                 const int32_t* kv_indptr, int32_t* kv_indices, cudaStream_t st) {
  if (N <= 0) return cudaSuccess;
  const int blocks = N < 65535 ? N : 65535;
  return launch_pdl(build_scatter_kernel, dim3(blocks), dim3(kTokThreads), 0, st, state_slot,
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
  cudaError_t e = launch_build_len(state_slot, swa_len, swa_head, comp_indptr, comp_block,
                                   comp_slot, comp_total, N, win, k_per_block, swa_pages,
                                   total_pages, kv_indptr, st);
  if (e == cudaSuccess)
    e = launch_pdl(build_scan_kernel, dim3(1), dim3(kScanThreads), 0, st, N, capacity, kv_indptr,
                   status);
  if (e == cudaSuccess)
    e = launch_build_scatter(state_slot, swa_len, swa_head, comp_indptr, comp_block, comp_slot, N,
                             win, k_per_block, swa_pages, kv_indptr, kv_indices, st);
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
