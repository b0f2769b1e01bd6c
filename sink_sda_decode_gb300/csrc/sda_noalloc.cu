// sda_noalloc.cu -- sda_decode_noalloc: the decode with its scratch memory
// in a fixed device array owned by this library, for callers that cannot
// allocate device memory themselves.
//
// Some hosts hand an operator nothing but its input and output buffers and
// forbid it to allocate (an inference engine that owns all device memory
// under a fixed budget, or a plain C caller without a device allocator).
// For them this entry point takes the same arguments as sda_decode minus the
// workspace, and uses `g_decode_scratch` below instead.
#include <cuda_runtime.h>

#include <mutex>

#include "sda_internal.cuh"

namespace sda {
namespace {

// The scratch array.  Every GPU that loads this library holds it until the
// process exits.  In host code the name is only a host-side stand-in: its
// device address comes from cudaGetSymbolAddress (below).
static __device__ __align__(256) unsigned char g_decode_scratch[SDA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

struct ScratchAddress {
  std::once_flag once;
  void* ptr = nullptr;
  cudaError_t err = cudaSuccess;
};
ScratchAddress g_scratch_address[kMaxDevices];

// Device address of the scratch array on the current device, looked up once
// per device with that device current.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  ScratchAddress& s = g_scratch_address[dev];
  std::call_once(s.once, [&]() { s.err = cudaGetSymbolAddress(&s.ptr, g_decode_scratch); });
  if (s.err != cudaSuccess) return s.err;
  if (s.ptr == nullptr) return cudaErrorInvalidSymbol;
  *out = s.ptr;
  return cudaSuccess;
}

}  // namespace
}  // namespace sda

extern "C" sda_status sda_decode_noalloc(const void* q, const void* unified_kv,
                                         int64_t total_pages, const int32_t* kv_indices,
                                         int64_t total_indices, const int32_t* kv_indptr,
                                         const float* attn_sink, float softmax_scale, int N, int H,
                                         int D, void* out, void* stream) {
  if (N < 0 || total_indices < 0) return SDA_ERR_INVALID_ARG;
  size_t need = 0;
  sda_status st = sda_decode_workspace_size(N, H, D, total_indices, &need);
  if (st != SDA_OK) return st;
  if (need > SDA_NOALLOC_SCRATCH_BYTES) return SDA_ERR_WORKSPACE;  // too big for the fixed array
  void* scratch = nullptr;
  if (sda::scratch_address(&scratch) != cudaSuccess) return SDA_ERR_CUDA;
  return sda_decode(q, unified_kv, total_pages, kv_indices, total_indices, kv_indptr, attn_sink,
                    softmax_scale, N, H, D, out, scratch, SDA_NOALLOC_SCRATCH_BYTES, stream);
}
