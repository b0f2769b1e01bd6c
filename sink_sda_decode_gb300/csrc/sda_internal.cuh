// sda_internal.cuh -- shared definitions of libsda's CUDA translation units:
// the workspace layout, the work-unit descriptor and the kernel launchers.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "sda.h"  // include/sda.h (on the include path of the build)

namespace sda {

// ---------------------------------------------------------------- work units
//
// A work unit is one piece of one token's slot list, for one group of heads.
// Each CTA of the persistent grid owns a contiguous run of units covering
// about the same number of KV tiles (the plan cuts each head group's tile
// sequence into equal ranges, "split-L"); the pieces of a token cut by a
// range boundary each write an unnormalised partial (m, l, acc) that the
// combine kernel merges with the sink.  Unsplit tokens are finished by the
// decode kernel.
//
// int4 layout: x = token, y = first index into kv_indices (absolute),
//              z = number of slots, w = head_group | ((partial_row + 1) << 4)
//              (partial_row + 1 == 0: the unit owns the whole token).
struct UnitDesc {
  int token, begin, len, meta;
};
__host__ __device__ inline int unit_head_group(int meta) { return meta & 15; }
__host__ __device__ inline int unit_part_row(int meta) { return (meta >> 4) - 1; }
__host__ __device__ inline int make_unit_meta(int head_group, int part_row) {
  return head_group | ((part_row + 1) << 4);
}

// Workspace header (first 256 bytes of the workspace).
struct WsHeader {
  int n_units;   // number of valid UnitDesc entries
  int n_split;   // number of split tokens (entries of the split list)
  int n_parts;   // partial rows in use
  int chunk;     // slots per piece chosen by the plan
  int error;     // nonzero: a pipeline wait timed out
  int pad[59];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

// Split list entry: x = token, y = first partial row, z = number of pieces.
constexpr int kTileSlots = 64;      // slots per KV tile of the tensor-core kernel
constexpr int kMaxPlanGrid = 1024;  // largest persistent grid the plan partitions for

// Decode variants.
enum Variant : int { kSimt = 0, kUmma = 1 };

struct LaunchPlan {
  Variant variant;
  int nh;        // heads per CTA
  int num_sms;   // SMs of the device
  int hg;        // head groups per token (H / nh)
  int grid;      // persistent CTAs the units are spread over
  int threads;   // threads per CTA
  size_t smem;   // dynamic shared memory bytes
  int tile;      // pieces of split lists are multiples of this many slots
};

struct WsLayout {
  // units_off: the unit list; cta_off: int [grid + 1], CTA b's units are
  // [cta[b], cta[b+1]); ctok_off / ctp_off: the plan's scratch (int [N], [N+1])
  size_t units_off, cta_off, ctok_off, ctp_off, split_off, ml_off, o_off, total;
  int u_max, s_max, p_max;
};

// What the plan needs to know about the device.
struct DeviceCaps {
  int num_sms = 0;
};
// The current device's capabilities (queried once per device).
cudaError_t device_caps(DeviceCaps* caps);

// Picks the kernel variant and grid for (H, D) on a device.  Returns false
// if (H, D) is unsupported.
bool choose_plan(int H, int D, const DeviceCaps& caps, LaunchPlan* lp);

// Workspace layout for a plan.  p_max bounds the partial rows: each of the
// at most grid / hg - 1 interior range boundaries cuts one token, so the
// split tokens have fewer than 2 * grid / hg pieces in total (and no more
// than one per tile).
WsLayout workspace_layout(int N, int H, int D, int64_t total_indices, const LaunchPlan& lp);

// ---------------------------------------------------------------- launchers
// All launchers only enqueue; they return cudaGetLastError().
cudaError_t launch_plan(const int32_t* kv_indptr, int N, int64_t total_indices,
                        const LaunchPlan& lp, void* ws, const WsLayout& L, cudaStream_t st);
// The builder's scan and the work plan in one CTA (sda_build_decode).
// Where the length pass left its findings on the compressed entries.  That
// pass checks the entry array in equal slices of chunks_per_cta 4-entry
// chunks, one slice per CTA, without knowing which token an entry belongs
// to, and writes flags[b] != 0 if slice b holds a bad entry; the tokens'
// lengths it writes assume good entries.  The scan then re-checks, entry by
// entry, every token whose entries overlap a flagged slice.
struct EntryCheck {
  const int32_t* state_slot;
  const int32_t* comp_indptr;
  const int32_t* comp_block;
  const int32_t* comp_slot;
  int64_t comp_total;
  int k_per_block;
  int64_t swa_pages;
  int64_t total_pages;
  const int32_t* flags;  // [n_flags]
  int n_flags;
  int64_t chunks_per_cta;
};

struct ScatterArgs;  // sda_scatter.cuh
// The work plan beside the index builder's scatter, one launch (after the
// builder's scan).
cudaError_t launch_scatter_plan(const ScatterArgs& sa, int64_t capacity, const LaunchPlan& lp,
                               void* ws, const WsLayout& L, int num_sms, cudaStream_t st);
cudaError_t launch_combine(const float* attn_sink, int N, int H, int D, void* out, void* ws,
                           const WsLayout& L, int num_sms, cudaStream_t st);
cudaError_t launch_decode_simt(const void* q, const void* kv, const int32_t* kv_indices,
                               const float* attn_sink, float softmax_scale, int N, int H, int D,
                               void* out, void* ws, const WsLayout& L, const LaunchPlan& lp,
                               cudaStream_t st);
// kv_scale == nullptr: kv is the bf16 pool; otherwise kv holds E4M3 codes
// [total_pages, D] and kv_scale [total_pages] the rows' dequantisation scales.
cudaError_t launch_decode_umma(const void* q, const void* kv, const float* kv_scale,
                               int64_t total_pages, const int32_t* kv_indices,
                               const float* attn_sink, float softmax_scale, int N, int H, int D,
                               void* out, void* ws, const WsLayout& L, const LaunchPlan& lp,
                               cudaStream_t st);
size_t umma_smem_bytes(int nh);
// Bound of the tensor-core kernel's pipeline waits, and whether CTA 0's
// first loader warp withholds one arrive (sda_debug_wait_fault; tests only).
struct WaitFault {
  int withhold;
  uint64_t timeout_ns;
};
WaitFault current_wait_fault();
cudaError_t umma_prepare(int nh);  // one-time kernel attribute set-up

cudaError_t launch_build_indices(const int32_t* state_slot, const int32_t* swa_len,
                                 const int32_t* swa_head, const int32_t* comp_indptr,
                                 const int32_t* comp_block, const int32_t* comp_slot,
                                 int64_t comp_total, int N, int win, int k_per_block,
                                 int64_t swa_pages, int64_t total_pages, int32_t* kv_indices,
                                 int64_t capacity, int32_t* kv_indptr, int32_t* status,
                                 cudaStream_t st);

// The layout of the length pass's entry check: its grid (one flag per CTA),
// its slices, and where the flags go (kv_indices, or the status word).
EntryCheck entry_check_layout(const int32_t* state_slot, const int32_t* comp_indptr,
                              const int32_t* comp_block, const int32_t* comp_slot,
                              int64_t comp_total, int N, int k_per_block, int64_t swa_pages,
                              int64_t total_pages, int64_t capacity, int32_t* kv_indices,
                              int32_t* status, int num_sms);
// The index builder as separate launches, for callers that put another
// kernel between its scan and its scatter: lengths and the entry check, then
// (after the scan, which takes the same EntryCheck) the scatter.
cudaError_t launch_build_len(const int32_t* swa_len, const int32_t* swa_head, int N, int win,
                             int32_t* kv_indptr, const EntryCheck& ec, cudaStream_t st);
cudaError_t launch_build_scan(int N, int64_t capacity, int32_t* kv_indptr, int32_t* status,
                              const EntryCheck& ec, cudaStream_t st);
cudaError_t launch_build_scatter(const int32_t* state_slot, const int32_t* swa_len,
                                 const int32_t* swa_head, const int32_t* comp_indptr,
                                 const int32_t* comp_block, const int32_t* comp_slot, int N,
                                 int win, int k_per_block, int64_t swa_pages, int64_t capacity,
                                 const int32_t* kv_indptr, int32_t* kv_indices, cudaStream_t st);
cudaError_t launch_validate(const int32_t* kv_indices, int64_t total_indices,
                            const int32_t* kv_indptr, int N, int64_t total_pages,
                            int32_t* status, cudaStream_t st);
// Top-k of each token's scores -> (comp_indptr, comp_block, comp_slot); the
// caller zeroes *status beforehand.
cudaError_t launch_topk_slots(const float* scores, int64_t score_stride, const int32_t* lengths,
                              const int32_t* block_table, int64_t bt_stride, int N, int k,
                              int k_per_block, int32_t* comp_indptr, int32_t* comp_block,
                              int32_t* comp_slot, int64_t capacity, int32_t* status,
                              cudaStream_t st);
// q/kv RMSNorm + RoPE + SWA ring store; bf16 pool when pool_fp8 == nullptr,
// else E4M3 codes + row scales.  The caller zeroes *status beforehand.
cudaError_t launch_qk_norm_rope_store(const void* q, const void* kv, const void* q_norm_w,
                                      const void* kv_norm_w, const float* cos_cache,
                                      const float* sin_cache, int max_pos,
                                      const int32_t* positions, const int32_t* state_slot, int N,
                                      int H, int D, int R, float eps, int win, int64_t swa_pages,
                                      void* q_out, void* pool, uint8_t* pool_fp8,
                                      float* pool_scale, int32_t* status, int num_sms,
                                      cudaStream_t st);

// Launch with programmatic dependent launch (PDL): the kernel may start while
// the previous kernel on the stream is still running (once that kernel has
// executed griddepcontrol.launch_dependents or exited).  Every kernel of this
// library calls pdl_wait() before its first global-memory access, which
// waits for the previous grid to complete and its writes to be visible, so
// only prologues (barrier init, TMEM allocation, descriptor prefetch)
// overlap.  Also valid inside CUDA-graph capture.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---------------------------------------------------------------- device helpers
#ifdef __CUDACC__
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ float ex2_approx(float x) {
  // hardware base-2 exponential (MUFU.EX2); ex2(-inf) = +0
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
constexpr float kLog2e = 1.4426950408889634f;

#endif

}  // namespace sda
