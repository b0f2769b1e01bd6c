// sda_build.cu -- the decode index builder and the index validator.
//
// The builder packs, per token, its SWA ring slots (state_slot * win + ring)
// and its compressed-cache slots (swa_pages + block_id * K_PER_BLOCK +
// slot_in_block) into the ragged kv_indices / kv_indptr pair the decode
// kernel reads (paged_decode.py docstring, caller convention for unified_kv
// and kv_indices: ragged-packed, no sentinels, padded tokens get an empty
// slice).  Three launches: lengths and an entry check (flat over the tokens
// and the compressed entries), a one-CTA scan (which re-checks the tokens
// whose entries were flagged), and the scatter.  Bad descriptors never reach
// the decode kernel: the token's slice is emptied and a status bit is raised
// (a divide-by-zero in a slot translation that produced out-of-range slots
// and a GPU fault is the failure the sglang PR 25898 summary page
// describes; here win and k_per_block are checked on the host and every
// emitted slot is in range).
#include "sda_internal.cuh"
#include "sda_scan.cuh"
#include "sda_scatter.cuh"

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

// Scatter pass (bodies in sda_scatter.cuh): one-token CTAs for a batch that
// fits one wave of them, else flat over the packed output.
constexpr int kScatterThreads = 256;

__global__ void __launch_bounds__(kTokThreads) build_scatter_tok_kernel(ScatterArgs a) {
  pdl_wait();
  pdl_trigger();
  scatter_tok_body(a, blockIdx.x, gridDim.x);
}

__global__ void __launch_bounds__(kScatterThreads) build_scatter_kernel(ScatterArgs a) {
  extern __shared__ int32_t s_ptr[];
  pdl_wait();
  pdl_trigger();
  scatter_flat_body(a, blockIdx.x, gridDim.x, s_ptr);
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

cudaError_t launch_build_scan(int N, int64_t capacity, int32_t* kv_indptr, int32_t* status,
                              const EntryCheck& ec, cudaStream_t st) {
  return launch_pdl(build_scan_kernel, dim3(1), dim3(kScanThreads), 0, st, N, capacity, kv_indptr,
                    status, ec);
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
  const ScatterArgs a{state_slot, swa_len, swa_head, comp_indptr, comp_block, comp_slot, N, win,
                      k_per_block, swa_pages, kv_indptr, kv_indices};
  const ScatterShape sh = scatter_shape(N, capacity, caps.num_sms, kScatterThreads);
  if (!sh.flat)
    return launch_pdl(build_scatter_tok_kernel, dim3(sh.ctas), dim3(kTokThreads), 0, st, a);
  return launch_pdl(build_scatter_kernel, dim3(sh.ctas), dim3(kScatterThreads), sh.smem, st, a);
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
  if (e == cudaSuccess) e = launch_build_scan(N, capacity, kv_indptr, status, ec, st);
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
