// sda_host.cu -- moving a step's inputs and result between page-locked host
// memory and the device with the SMs instead of the copy engines.
//
// A decode step's host traffic is small (q and the index descriptors in, out
// back: about 2 MB for 64 tokens of 16 heads), so a copy-engine transfer is
// dominated by its fixed latency.  Page-locked host memory is addressable
// from kernels (unified addressing; over NVLink-C2C on Grace-based systems),
// so one grid-stride kernel gathers every input array into the device
// workspace and another writes the result back, each a PDL-chained launch
// inside the same CUDA graph as the step.
#include <cuda_runtime.h>

#include <cstdint>

#include "sda_copy.cuh"
#include "sda_internal.cuh"

namespace sda {

namespace {

constexpr int kCopyThreads = 256;

// Segments are 4-byte aligned with sizes in 4-byte words; a segment whose
// ends are both 16-byte aligned moves its whole 16-byte part with uint4.
__global__ void __launch_bounds__(kCopyThreads) gather_copy_kernel(CopySegments segs) {
  pdl_wait();
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * kCopyThreads + threadIdx.x;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kCopyThreads;
  for (int i = 0; i < segs.n; ++i) {
    const CopySegment& s = segs.seg[i];
    const uint32_t* src = static_cast<const uint32_t*>(s.src);
    uint32_t* dst = static_cast<uint32_t*>(s.dst);
    int64_t done = 0;
    if (((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 15) == 0) {
      const int64_t n16 = s.words / 4;
      const uint4* s4 = reinterpret_cast<const uint4*>(src);
      uint4* d4 = reinterpret_cast<uint4*>(dst);
      for (int64_t k = tid; k < n16; k += stride) d4[k] = s4[k];
      done = n16 * 4;
    }
    for (int64_t k = done + tid; k < s.words; k += stride) dst[k] = src[k];
  }
  pdl_trigger();
}

}  // namespace

cudaError_t launch_gather_copy(const CopySegments& segs, int num_sms, cudaStream_t st) {
  int64_t words = 0;
  for (int i = 0; i < segs.n; ++i) words += segs.seg[i].words;
  if (words == 0) return cudaSuccess;
  // enough CTAs for one 16-byte load per thread, at most 4 per SM
  const int64_t want = (words / 4 + kCopyThreads - 1) / kCopyThreads + 1;
  const int64_t cap = static_cast<int64_t>(num_sms) * 4;
  const int grid = static_cast<int>(want < cap ? want : cap);
  return launch_pdl(gather_copy_kernel, dim3(grid), dim3(kCopyThreads), 0, st, segs);
}

}  // namespace sda
