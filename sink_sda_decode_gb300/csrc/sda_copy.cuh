// sda_copy.cuh -- the gather-copy launch that moves a step's inputs and
// result between page-locked host memory and the device (sda_host.cu), used
// by sda_build_decode_host.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace sda {

// Copies between arrays the SMs can address (device memory, page-locked host
// memory), in one grid-stride launch; every segment 4-byte aligned.
struct CopySegment {
  const void* src;
  void* dst;
  int64_t words;  // 4-byte words
};
constexpr int kMaxCopySegments = 8;
struct CopySegments {
  CopySegment seg[kMaxCopySegments];
  int n;
};
cudaError_t launch_gather_copy(const CopySegments& segs, int num_sms, cudaStream_t st);

}  // namespace sda
