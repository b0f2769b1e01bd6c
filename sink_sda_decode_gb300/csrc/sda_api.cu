// sda_api.cu -- the extern "C" entry points of libsda (declared in
// include/sda.h): host-side argument checks, kernel-variant choice, the
// workspace layout, and the launches.  Nothing here allocates, synchronises
// or reads device memory from the host.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "sda_copy.cuh"
#include "sda_internal.cuh"
#include "sda_scatter.cuh"

namespace sda {

namespace {

thread_local char g_last_error[256] = "";
// sda_debug_wait_fault: pipeline-wait bound (0 = the default 2 s) and the
// withheld-arrive switch, read by every tensor-core kernel launch.
std::atomic<unsigned long long> g_wait_timeout_ns{0};
std::atomic<int> g_withhold_arrive{0};
constexpr unsigned long long kDefaultWaitTimeoutNs = 2000000000ull;
thread_local cudaEvent_t g_ev_before = nullptr;
thread_local cudaEvent_t g_ev_after = nullptr;

void note_cuda_error(cudaError_t e, const char* where) {
  std::snprintf(g_last_error, sizeof g_last_error, "%s: %s (%s)", where, cudaGetErrorName(e),
                cudaGetErrorString(e));
}

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  std::once_flag once;
  DeviceCaps caps;
  cudaError_t err = cudaSuccess;
};
DeviceInfo g_dev[kMaxDevices];

}  // namespace

// SM count of the current device, queried once per device; also sets the
// tensor-core kernels' shared-memory attributes on that device.
cudaError_t device_caps(DeviceCaps* caps) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  DeviceInfo& d = g_dev[dev];
  std::call_once(d.once, [&]() {
    d.err = cudaDeviceGetAttribute(&d.caps.num_sms, cudaDevAttrMultiProcessorCount, dev);
    for (int nh : {16, 32, 64})
      if (d.err == cudaSuccess) d.err = umma_prepare(nh);
  });
  *caps = d.caps;
  return d.err;
}

namespace {

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Optional A/B switch for tests: SDA_FORCE_VARIANT=simt|umma forces a
// decode kernel (umma only where the shape allows it).
int forced_variant() {
  const char* v = std::getenv("SDA_FORCE_VARIANT");
  if (!v) return -1;
  if (std::strcmp(v, "simt") == 0) return kSimt;
  if (std::strcmp(v, "umma") == 0) return kUmma;
  return -1;
}

}  // namespace

WaitFault current_wait_fault() {
  const unsigned long long t = g_wait_timeout_ns.load();
  return WaitFault{g_withhold_arrive.load(), t ? t : kDefaultWaitTimeoutNs};
}

bool shape_supported(int H, int D) {
  return (D == 64 || D == 128 || D == 256 || D == 512) && H >= 1 && H <= 256;
}

bool tc_shape_supported(int H, int D) {
  return D == 512 && (H == 16 || H == 32 || (H % 64 == 0 && H <= 256));
}

bool choose_plan(int H, int D, const DeviceCaps& caps, LaunchPlan* lp) {
  if (!shape_supported(H, D)) return false;
  lp->num_sms = caps.num_sms;
  const bool tc_shape = tc_shape_supported(H, D);
  const int nh = H < 64 ? H : 64;
  const int forced = forced_variant();
  Variant v = tc_shape ? kUmma : kSimt;
  if (forced == kSimt || (forced == kUmma && tc_shape)) v = static_cast<Variant>(forced);
  lp->variant = v;
  if (v == kUmma) {
    lp->nh = nh;
    lp->hg = H / lp->nh;
    lp->grid = caps.num_sms;  // one CTA per SM (about 200 KB of shared memory each)
    lp->threads = 896;
    lp->smem = umma_smem_bytes(lp->nh);
    lp->tile = kTileSlots;
  } else {
    lp->nh = H;
    lp->hg = 1;
    lp->grid = caps.num_sms * 4;
    lp->threads = 256;
    lp->smem = 0;
    lp->tile = kTileSlots;
  }
  if (lp->grid > kMaxPlanGrid) lp->grid = kMaxPlanGrid;
  return true;
}

WsLayout workspace_layout(int N, int H, int D, int64_t total_indices, const LaunchPlan& lp) {
  WsLayout L;
  // Partial rows: fewer than 2 * grid / hg (each interior range boundary
  // cuts one token) and no more than one per tile (T <= total_indices).
  int64_t p1 = 2 * ((int64_t)(lp.grid + lp.hg - 1) / lp.hg) + 2;
  int64_t p2 = 2 * ((total_indices + lp.tile - 1) / lp.tile) + 2;
  int64_t p_max = p1 < p2 ? p1 : p2;
  int64_t s_max = p_max / 2 + 1;
  if (s_max > N) s_max = N;
  L.p_max = (int)p_max;
  L.s_max = (int)s_max;
  L.u_max = (int)((int64_t)lp.hg * ((int64_t)N + p_max));
  size_t off = sizeof(WsHeader);
  L.units_off = off;
  off = align_up(off + (size_t)L.u_max * 16, 256);
  L.cta_off = off;
  off = align_up(off + (size_t)(lp.grid + 1) * 4, 256);
  L.ctok_off = off;
  off = align_up(off + (size_t)(N > 0 ? N : 1) * 4, 256);
  L.ctp_off = off;
  off = align_up(off + (size_t)(N + 1) * 4, 256);
  L.split_off = off;
  off = align_up(off + (size_t)(s_max > 0 ? s_max : 1) * 16, 256);
  L.ml_off = off;
  off = align_up(off + (size_t)p_max * H * 8, 256);
  L.o_off = off;
  off = align_up(off + (size_t)p_max * H * D * 4, 256);
  L.total = off;
  return L;
}

}  // namespace sda

using namespace sda;

extern "C" {

const char* sda_strerror(sda_status status) {
  switch (status) {
    case SDA_OK: return "SDA_OK";
    case SDA_ERR_INVALID_ARG: return "SDA_ERR_INVALID_ARG: invalid argument";
    case SDA_ERR_UNSUPPORTED: return "SDA_ERR_UNSUPPORTED: unsupported (H, D)";
    case SDA_ERR_CUDA: return "SDA_ERR_CUDA: a CUDA call failed";
    case SDA_ERR_WORKSPACE: return "SDA_ERR_WORKSPACE: workspace too small or misaligned";
    default: return "SDA: unknown status";
  }
}

const char* sda_last_cuda_error(void) { return g_last_error; }

int sda_abi_version(void) { return 1; }

sda_status sda_decode_workspace_size(int N, int H, int D, int64_t total_indices, size_t* bytes) {
  if (!bytes || N < 0 || total_indices < 0) return SDA_ERR_INVALID_ARG;
  if (!shape_supported(H, D)) return SDA_ERR_UNSUPPORTED;
  DeviceCaps caps;
  cudaError_t e = device_caps(&caps);
  if (e != cudaSuccess) {
    note_cuda_error(e, "sda_decode_workspace_size");
    return SDA_ERR_CUDA;
  }
  LaunchPlan lp;
  if (!choose_plan(H, D, caps, &lp)) return SDA_ERR_UNSUPPORTED;
  *bytes = workspace_layout(N, H, D, total_indices, lp).total;
  return SDA_OK;
}

sda_status sda_decode(const void* q, const void* unified_kv, int64_t total_pages,
                      const int32_t* kv_indices, int64_t total_indices,
                      const int32_t* kv_indptr, const float* attn_sink, float softmax_scale,
                      int N, int H, int D, void* out, void* workspace, size_t workspace_bytes,
                      void* stream) {
  if (N < 0 || total_indices < 0 || total_indices > 0x7fffffffll) return SDA_ERR_INVALID_ARG;
  if (total_pages <= 0 || total_pages > 0x7fffffffll) return SDA_ERR_INVALID_ARG;
  if (!shape_supported(H, D)) return SDA_ERR_UNSUPPORTED;
  if (N == 0) return SDA_OK;
  if (!q || !unified_kv || !kv_indptr || !attn_sink || !out || !workspace) return SDA_ERR_INVALID_ARG;
  if (total_indices > 0 && !kv_indices) return SDA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(unified_kv, 16) || !aligned(out, 16) || !aligned(kv_indptr, 4) ||
      !aligned(attn_sink, 4) || (kv_indices && !aligned(kv_indices, 4)))
    return SDA_ERR_INVALID_ARG;
  if (!aligned(workspace, 256)) return SDA_ERR_WORKSPACE;
  DeviceCaps caps;
  cudaError_t e = device_caps(&caps);
  if (e != cudaSuccess) {
    note_cuda_error(e, "sda_decode");
    return SDA_ERR_CUDA;
  }
  LaunchPlan lp;
  choose_plan(H, D, caps, &lp);
  const WsLayout L = workspace_layout(N, H, D, total_indices, lp);
  if (workspace_bytes < L.total) return SDA_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  e = launch_plan(kv_indptr, N, total_indices, lp, workspace, L, st);
  if (e == cudaSuccess && g_ev_before && g_ev_after) e = cudaEventRecord(g_ev_before, st);
  if (e == cudaSuccess) {
    if (lp.variant == kUmma)
      e = launch_decode_umma(q, unified_kv, nullptr, total_pages, kv_indices, attn_sink,
                             softmax_scale, N, H, D, out, workspace, L, lp, st);
    else
      e = launch_decode_simt(q, unified_kv, kv_indices, attn_sink, softmax_scale, N, H, D, out,
                             workspace, L, lp, st);
  }
  if (e == cudaSuccess && g_ev_before && g_ev_after) e = cudaEventRecord(g_ev_after, st);
  if (e == cudaSuccess) e = launch_combine(attn_sink, N, H, D, out, workspace, L, caps.num_sms, st);
  if (e != cudaSuccess) {
    note_cuda_error(e, "sda_decode");
    return SDA_ERR_CUDA;
  }
  return SDA_OK;
}

// The FP8-pool entry points run the one-CTA tensor-core kernel only.
static bool fp8_plan(int H, int D, const DeviceCaps& caps, LaunchPlan* lp) {
  if (!tc_shape_supported(H, D) || !choose_plan(H, D, caps, lp)) return false;
  if (lp->variant != kUmma) {  // a forced variant does not apply to the FP8 pool
    lp->variant = kUmma;
    lp->nh = H < 64 ? H : 64;
    lp->hg = H / lp->nh;
    lp->grid = caps.num_sms;
    lp->threads = 896;
    lp->smem = umma_smem_bytes(lp->nh);
    lp->tile = kTileSlots;
  }
  return true;
}

sda_status sda_decode_fp8_workspace_size(int N, int H, int D, int64_t total_indices, size_t* bytes) {
  if (!bytes || N < 0 || total_indices < 0) return SDA_ERR_INVALID_ARG;
  if (!tc_shape_supported(H, D)) return SDA_ERR_UNSUPPORTED;
  DeviceCaps caps;
  cudaError_t e = device_caps(&caps);
  if (e != cudaSuccess) {
    note_cuda_error(e, "sda_decode_fp8_workspace_size");
    return SDA_ERR_CUDA;
  }
  LaunchPlan lp;
  if (!fp8_plan(H, D, caps, &lp)) return SDA_ERR_UNSUPPORTED;
  *bytes = workspace_layout(N, H, D, total_indices, lp).total;
  return SDA_OK;
}

sda_status sda_decode_fp8(const void* q, const void* kv_fp8, const float* kv_scale,
                          int64_t total_pages, const int32_t* kv_indices, int64_t total_indices,
                          const int32_t* kv_indptr, const float* attn_sink, float softmax_scale,
                          int N, int H, int D, void* out, void* workspace, size_t workspace_bytes,
                          void* stream) {
  if (N < 0 || total_indices < 0 || total_indices > 0x7fffffffll) return SDA_ERR_INVALID_ARG;
  if (total_pages <= 0 || total_pages > 0x7fffffffll) return SDA_ERR_INVALID_ARG;
  if (!tc_shape_supported(H, D)) return SDA_ERR_UNSUPPORTED;
  if (N == 0) return SDA_OK;
  if (!q || !kv_fp8 || !kv_scale || !kv_indptr || !attn_sink || !out || !workspace)
    return SDA_ERR_INVALID_ARG;
  if (total_indices > 0 && !kv_indices) return SDA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(kv_fp8, 16) || !aligned(out, 16) || !aligned(kv_scale, 4) ||
      !aligned(kv_indptr, 4) || !aligned(attn_sink, 4) || (kv_indices && !aligned(kv_indices, 4)))
    return SDA_ERR_INVALID_ARG;
  if (!aligned(workspace, 256)) return SDA_ERR_WORKSPACE;
  DeviceCaps caps;
  cudaError_t e = device_caps(&caps);
  if (e != cudaSuccess) {
    note_cuda_error(e, "sda_decode_fp8");
    return SDA_ERR_CUDA;
  }
  LaunchPlan lp;
  fp8_plan(H, D, caps, &lp);
  const WsLayout L = workspace_layout(N, H, D, total_indices, lp);
  if (workspace_bytes < L.total) return SDA_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  e = launch_plan(kv_indptr, N, total_indices, lp, workspace, L, st);
  if (e == cudaSuccess && g_ev_before && g_ev_after) e = cudaEventRecord(g_ev_before, st);
  if (e == cudaSuccess)
    e = launch_decode_umma(q, kv_fp8, kv_scale, total_pages, kv_indices, attn_sink, softmax_scale,
                           N, H, D, out, workspace, L, lp, st);
  if (e == cudaSuccess && g_ev_before && g_ev_after) e = cudaEventRecord(g_ev_after, st);
  if (e == cudaSuccess) e = launch_combine(attn_sink, N, H, D, out, workspace, L, caps.num_sms, st);
  if (e != cudaSuccess) {
    note_cuda_error(e, "sda_decode_fp8");
    return SDA_ERR_CUDA;
  }
  return SDA_OK;
}

// The scalar and pool-argument checks of sda_build_decode(_host) that need
// no workspace-derived pointer; the host-buffer entry point runs them before
// it enqueues its input gather, so that an invalid call enqueues nothing.
static sda_status build_decode_scalars_ok(int N, int win, int k_per_block, int64_t swa_pages,
                                          int64_t total_pages, int64_t capacity,
                                          int64_t comp_total, const void* unified_kv,
                                          const float* kv_scale, const float* attn_sink, int H,
                                          int D) {
  if (N < 0 || win <= 0 || k_per_block <= 0 || swa_pages < 0 || total_pages <= 0 ||
      total_pages > 0x7fffffffll || swa_pages > total_pages || capacity < 0 ||
      capacity > 0x7fffffffll || comp_total < 0 || comp_total > 0x7fffffffll)
    return SDA_ERR_INVALID_ARG;
  const bool fp8 = kv_scale != nullptr;
  if (fp8 ? !tc_shape_supported(H, D) : !shape_supported(H, D)) return SDA_ERR_UNSUPPORTED;
  if (N > 0 && (!unified_kv || !attn_sink || !aligned(unified_kv, 16) || !aligned(attn_sink, 4) ||
                (fp8 && !aligned(kv_scale, 4))))
    return SDA_ERR_INVALID_ARG;
  return SDA_OK;
}

static sda_status build_decode_impl(const int32_t* state_slot, const int32_t* swa_len,
                                    const int32_t* swa_head, const int32_t* comp_indptr,
                                    const int32_t* comp_block, const int32_t* comp_slot,
                                    int64_t comp_total, int win, int k_per_block,
                                    int64_t swa_pages, int32_t* kv_indices, int64_t capacity,
                                    int32_t* kv_indptr, int32_t* status, const void* q,
                                    const void* unified_kv, const float* kv_scale,
                                    int64_t total_pages, const float* attn_sink,
                                    float softmax_scale, int N, int H, int D, void* out,
                                    void* workspace, size_t workspace_bytes, void* stream,
                                    const char* who) {
  // the builder's checks (sda_build_indices)
  if (N < 0 || win <= 0 || k_per_block <= 0 || swa_pages < 0 || total_pages <= 0 ||
      total_pages > 0x7fffffffll || swa_pages > total_pages || capacity < 0 ||
      capacity > 0x7fffffffll || comp_total < 0 || comp_total > 0x7fffffffll)
    return SDA_ERR_INVALID_ARG;
  if (!kv_indptr || !status) return SDA_ERR_INVALID_ARG;
  if (N > 0 && (!state_slot || !swa_len || !swa_head || !comp_indptr)) return SDA_ERR_INVALID_ARG;
  if (comp_total > 0 && (!comp_block || !comp_slot)) return SDA_ERR_INVALID_ARG;
  if (capacity > 0 && !kv_indices) return SDA_ERR_INVALID_ARG;
  // the decode's checks (sda_decode / sda_decode_fp8)
  const bool fp8 = kv_scale != nullptr;
  if (fp8 ? !tc_shape_supported(H, D) : !shape_supported(H, D)) return SDA_ERR_UNSUPPORTED;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (N == 0) {  // the builder still writes kv_indptr[0] and the status word
    const cudaError_t e = launch_build_indices(state_slot, swa_len, swa_head, comp_indptr,
                                               comp_block, comp_slot, comp_total, N, win,
                                               k_per_block, swa_pages, total_pages, kv_indices,
                                               capacity, kv_indptr, status, st);
    if (e != cudaSuccess) {
      note_cuda_error(e, who);
      return SDA_ERR_CUDA;
    }
    return SDA_OK;
  }
  if (!q || !unified_kv || !attn_sink || !out || !workspace) return SDA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(unified_kv, 16) || !aligned(out, 16) || !aligned(kv_indptr, 4) ||
      !aligned(attn_sink, 4) || (kv_indices && !aligned(kv_indices, 4)) ||
      (fp8 && !aligned(kv_scale, 4)))
    return SDA_ERR_INVALID_ARG;
  if (!aligned(workspace, 256)) return SDA_ERR_WORKSPACE;
  DeviceCaps caps;
  cudaError_t e = device_caps(&caps);
  if (e != cudaSuccess) {
    note_cuda_error(e, who);
    return SDA_ERR_CUDA;
  }
  LaunchPlan lp;
  if (fp8) fp8_plan(H, D, caps, &lp);
  else choose_plan(H, D, caps, &lp);
  const WsLayout L = workspace_layout(N, H, D, capacity, lp);
  if (workspace_bytes < L.total) return SDA_ERR_WORKSPACE;
  const EntryCheck ec = entry_check_layout(state_slot, comp_indptr, comp_block, comp_slot,
                                           comp_total, N, k_per_block, swa_pages, total_pages,
                                           capacity, kv_indices, status, caps.num_sms);
  e = launch_build_len(swa_len, swa_head, N, win, kv_indptr, ec, st);
  if (e == cudaSuccess) e = launch_build_scan(N, capacity, kv_indptr, status, ec, st);
  if (e == cudaSuccess) {
    const ScatterArgs sa{state_slot, swa_len, swa_head, comp_indptr, comp_block, comp_slot, N, win,
                         k_per_block, swa_pages, kv_indptr, kv_indices};
    e = launch_scatter_plan(sa, capacity, lp, workspace, L, caps.num_sms, st);
  }
  if (e == cudaSuccess && g_ev_before && g_ev_after) e = cudaEventRecord(g_ev_before, st);
  if (e == cudaSuccess) {
    if (fp8)
      e = launch_decode_umma(q, unified_kv, kv_scale, total_pages, kv_indices, attn_sink,
                             softmax_scale, N, H, D, out, workspace, L, lp, st);
    else if (lp.variant == kUmma)
      e = launch_decode_umma(q, unified_kv, nullptr, total_pages, kv_indices, attn_sink,
                             softmax_scale, N, H, D, out, workspace, L, lp, st);
    else
      e = launch_decode_simt(q, unified_kv, kv_indices, attn_sink, softmax_scale, N, H, D, out,
                             workspace, L, lp, st);
  }
  if (e == cudaSuccess && g_ev_before && g_ev_after) e = cudaEventRecord(g_ev_after, st);
  if (e == cudaSuccess) e = launch_combine(attn_sink, N, H, D, out, workspace, L, caps.num_sms, st);
  if (e != cudaSuccess) {
    note_cuda_error(e, who);
    return SDA_ERR_CUDA;
  }
  return SDA_OK;
}

sda_status sda_build_decode(const int32_t* state_slot, const int32_t* swa_len,
                            const int32_t* swa_head, const int32_t* comp_indptr,
                            const int32_t* comp_block, const int32_t* comp_slot,
                            int64_t comp_total, int win, int k_per_block, int64_t swa_pages,
                            int32_t* kv_indices, int64_t capacity, int32_t* kv_indptr,
                            int32_t* status, const void* q, const void* unified_kv,
                            const float* kv_scale, int64_t total_pages, const float* attn_sink,
                            float softmax_scale, int N, int H, int D, void* out, void* workspace,
                            size_t workspace_bytes, void* stream) {
  return build_decode_impl(state_slot, swa_len, swa_head, comp_indptr, comp_block, comp_slot,
                           comp_total, win, k_per_block, swa_pages, kv_indices, capacity,
                           kv_indptr, status, q, unified_kv, kv_scale, total_pages, attn_sink,
                           softmax_scale, N, H, D, out, workspace, workspace_bytes, stream,
                           "sda_build_decode");
}

// Layout of sda_build_decode_host's device workspace: the staged inputs, the
// builder's outputs, the staged output, then sda_build_decode's workspace.
struct HostWs {
  size_t q, ss, sl, sh, cptr, cb, cs, idx, iptr, st, out, dec, total;
};

static HostWs host_ws_layout(int N, int H, int D, int64_t comp_total, int64_t capacity,
                             size_t dec_bytes) {
  HostWs w;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + (bytes > 0 ? bytes : 1), 256);
    return at;
  };
  const size_t qb = (size_t)N * H * D * 2;
  w.q = take(qb);
  w.ss = take((size_t)N * 4);
  w.sl = take((size_t)N * 4);
  w.sh = take((size_t)N * 4);
  w.cptr = take((size_t)(N + 1) * 4);
  w.cb = take((size_t)comp_total * 4);
  w.cs = take((size_t)comp_total * 4);
  w.idx = take((size_t)capacity * 4);
  w.iptr = take((size_t)(N + 1) * 4);
  w.st = take(4);
  w.out = take(qb);
  w.dec = take(dec_bytes);
  w.total = off;
  return w;
}

// Device view of page-locked host memory (NULL if `p` is not page-locked host memory).
static const void* host_view(const void* p) {
  if (!p) return nullptr;
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

static sda_status build_decode_ws(int N, int H, int D, int64_t capacity, bool fp8, size_t* bytes) {
  DeviceCaps caps;
  const cudaError_t e = device_caps(&caps);
  if (e != cudaSuccess) {
    note_cuda_error(e, "sda_build_decode_host_workspace_size");
    return SDA_ERR_CUDA;
  }
  LaunchPlan lp;
  if (fp8) fp8_plan(H, D, caps, &lp);
  else choose_plan(H, D, caps, &lp);
  *bytes = workspace_layout(N, H, D, capacity, lp).total;
  return SDA_OK;
}

// ---------------------------------------------------------------- large host batches
// A batch whose q (and out) is at least kPipelineBytes moves through the
// host link in token chunks so that the link's two directions and the SMs
// work at once: two streams of this library carry copy-engine transfers (the
// descriptors and each chunk's q in; each chunk's out back as soon as its
// decode is done) while the caller's stream builds the whole batch's lists
// once and decodes chunk after chunk (the decode takes absolute kv_indptr
// offsets, so a chunk decodes from a slice of the batch's lists).  The
// chunk boundaries depend on N only, never on the contents of the host
// arrays, so a captured graph stays valid when the caller refills them.
constexpr int64_t kPipelineBytes = 8ll << 20;
constexpr int kMaxChunks = 8;

struct PipeRes {
  cudaStream_t cin = nullptr, cout = nullptr;
  cudaEvent_t fork = nullptr, desc = nullptr, built = nullptr, done = nullptr;
  cudaEvent_t q_in[kMaxChunks] = {}, dec_done[kMaxChunks] = {};
  bool ok = false;
};

// Streams and events of the current device, created on its first large
// call (which should therefore come before any stream capture); calls that
// enqueue concurrently from several host threads are serialised.
static std::mutex g_pipe_mu;
static PipeRes g_pipe[64];

static cudaError_t pipe_resources(PipeRes** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  PipeRes& r = g_pipe[dev];
  if (!r.ok) {
    // all or nothing: a failure destroys whatever this attempt created
    PipeRes n;
    const unsigned fl = cudaEventDisableTiming;
    cudaEvent_t* evs[4 + 2 * kMaxChunks] = {&n.fork, &n.desc, &n.built, &n.done};
    for (int c = 0; c < kMaxChunks; ++c) {
      evs[4 + 2 * c] = &n.q_in[c];
      evs[5 + 2 * c] = &n.dec_done[c];
    }
    e = cudaStreamCreateWithFlags(&n.cin, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&n.cout, cudaStreamNonBlocking);
    for (cudaEvent_t* p : evs)
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(p, fl);
    if (e != cudaSuccess) {
      for (cudaEvent_t* p : evs)
        if (*p) cudaEventDestroy(*p);
      if (n.cin) cudaStreamDestroy(n.cin);
      if (n.cout) cudaStreamDestroy(n.cout);
      return e;
    }
    n.ok = true;
    r = n;
  }
  *out = &r;
  return cudaSuccess;
}

static sda_status build_decode_host_pipelined(
    const int32_t* state_slot, const int32_t* swa_len, const int32_t* swa_head,
    const int32_t* comp_indptr, const int32_t* comp_block, const int32_t* comp_slot,
    int64_t comp_total, int win, int k_per_block, int64_t swa_pages, int64_t capacity,
    const void* q, const void* unified_kv, const float* kv_scale, int64_t total_pages,
    const float* attn_sink, float softmax_scale, int N, int H, int D, void* out, int32_t* status,
    char* base, const HostWs& w, cudaStream_t st) {
  const char* who = "sda_build_decode_host";
  const bool fp8 = kv_scale != nullptr;
  DeviceCaps caps;
  cudaError_t e = device_caps(&caps);
  if (e != cudaSuccess) {
    note_cuda_error(e, who);
    return SDA_ERR_CUDA;
  }
  LaunchPlan lp;
  if (fp8) fp8_plan(H, D, caps, &lp);
  else choose_plan(H, D, caps, &lp);
  std::lock_guard<std::mutex> lock(g_pipe_mu);
  PipeRes* r = nullptr;
  e = pipe_resources(&r);
  const int64_t row_bytes = (int64_t)H * D * 2;  // q / out bytes per token
  const int64_t q_bytes = (int64_t)N * row_bytes;
  int chunks = (int)(q_bytes / kPipelineBytes);
  chunks = chunks < 2 ? 2 : (chunks > kMaxChunks ? kMaxChunks : chunks);
  if (chunks > N) chunks = N;
  const int per = (N + chunks - 1) / chunks;
  auto H2D = [&](void* dst, const void* src, size_t bytes) {
    return bytes ? cudaMemcpyAsync(dst, src, bytes, cudaMemcpyHostToDevice, r->cin) : cudaSuccess;
  };
  // fork: the copy streams start after everything already on the caller's stream
  if (e == cudaSuccess) e = cudaEventRecord(r->fork, st);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(r->cin, r->fork, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(r->cout, r->fork, 0);
  // descriptors, then the q chunks, on the inbound stream
  if (e == cudaSuccess) e = H2D(base + w.ss, state_slot, (size_t)N * 4);
  if (e == cudaSuccess) e = H2D(base + w.sl, swa_len, (size_t)N * 4);
  if (e == cudaSuccess) e = H2D(base + w.sh, swa_head, (size_t)N * 4);
  if (e == cudaSuccess) e = H2D(base + w.cptr, comp_indptr, (size_t)(N + 1) * 4);
  if (e == cudaSuccess) e = H2D(base + w.cb, comp_block, (size_t)comp_total * 4);
  if (e == cudaSuccess) e = H2D(base + w.cs, comp_slot, (size_t)comp_total * 4);
  if (e == cudaSuccess) e = cudaEventRecord(r->desc, r->cin);
  for (int c = 0; c < chunks && e == cudaSuccess; ++c) {
    const int t0 = c * per, nc = (t0 + per <= N ? per : N - t0);
    if (nc <= 0) break;
    e = H2D(base + w.q + (size_t)t0 * row_bytes, static_cast<const char*>(q) + (size_t)t0 * row_bytes,
            (size_t)nc * row_bytes);
    if (e == cudaSuccess) e = cudaEventRecord(r->q_in[c], r->cin);
  }
  // the whole batch's lists and status on the caller's stream
  int32_t* idx = reinterpret_cast<int32_t*>(base + w.idx);
  int32_t* iptr = reinterpret_cast<int32_t*>(base + w.iptr);
  int32_t* dst_st = reinterpret_cast<int32_t*>(base + w.st);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(st, r->desc, 0);
  if (e == cudaSuccess)
    e = launch_build_indices(reinterpret_cast<const int32_t*>(base + w.ss),
                             reinterpret_cast<const int32_t*>(base + w.sl),
                             reinterpret_cast<const int32_t*>(base + w.sh),
                             reinterpret_cast<const int32_t*>(base + w.cptr),
                             reinterpret_cast<const int32_t*>(base + w.cb),
                             reinterpret_cast<const int32_t*>(base + w.cs), comp_total, N, win,
                             k_per_block, swa_pages, total_pages, idx, capacity, iptr, dst_st, st);
  if (e == cudaSuccess) e = cudaEventRecord(r->built, st);
  // the status word goes back as soon as the build is done
  if (e == cudaSuccess) e = cudaStreamWaitEvent(r->cout, r->built, 0);
  if (e == cudaSuccess) e = cudaMemcpyAsync(status, dst_st, 4, cudaMemcpyDeviceToHost, r->cout);
  // decode chunk after chunk; each chunk's out goes back on the outbound stream
  void* dec = base + w.dec;
  for (int c = 0; c < chunks && e == cudaSuccess; ++c) {
    const int t0 = c * per, nc = (t0 + per <= N ? per : N - t0);
    if (nc <= 0) break;
    const WsLayout L = workspace_layout(nc, H, D, capacity, lp);
    const char* qc = base + w.q + (size_t)t0 * row_bytes;
    char* oc = base + w.out + (size_t)t0 * row_bytes;
    e = cudaStreamWaitEvent(st, r->q_in[c], 0);
    if (e == cudaSuccess) e = launch_plan(iptr + t0, nc, capacity, lp, dec, L, st);
    if (e == cudaSuccess) {
      if (fp8 || lp.variant == kUmma)
        e = launch_decode_umma(qc, unified_kv, kv_scale, total_pages, idx, attn_sink, softmax_scale,
                               nc, H, D, oc, dec, L, lp, st);
      else
        e = launch_decode_simt(qc, unified_kv, idx, attn_sink, softmax_scale, nc, H, D, oc, dec,
                               L, lp, st);
    }
    if (e == cudaSuccess) e = launch_combine(attn_sink, nc, H, D, oc, dec, L, caps.num_sms, st);
    if (e == cudaSuccess) e = cudaEventRecord(r->dec_done[c], st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(r->cout, r->dec_done[c], 0);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(static_cast<char*>(out) + (size_t)t0 * row_bytes, oc, (size_t)nc * row_bytes,
                          cudaMemcpyDeviceToHost, r->cout);
  }
  // join: the caller's stream continues after every copy of this call
  if (e == cudaSuccess) e = cudaEventRecord(r->done, r->cout);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(st, r->done, 0);
  if (e == cudaSuccess) e = cudaEventRecord(r->fork, r->cin);  // the inbound stream joins too
  if (e == cudaSuccess) e = cudaStreamWaitEvent(st, r->fork, 0);
  if (e != cudaSuccess) {
    note_cuda_error(e, who);
    return SDA_ERR_CUDA;
  }
  return SDA_OK;
}

sda_status sda_build_decode_host_workspace_size(int N, int H, int D, int64_t comp_total,
                                                int64_t capacity, int fp8, size_t* bytes) {
  if (!bytes || N < 0 || comp_total < 0 || capacity < 0) return SDA_ERR_INVALID_ARG;
  if (fp8 ? !tc_shape_supported(H, D) : !shape_supported(H, D)) return SDA_ERR_UNSUPPORTED;
  size_t dec = 0;
  const sda_status r = build_decode_ws(N, H, D, capacity, fp8 != 0, &dec);
  if (r != SDA_OK) return r;
  *bytes = host_ws_layout(N, H, D, comp_total, capacity, dec).total;
  if ((int64_t)N * H * D * 2 >= kPipelineBytes && N >= 2) {
    // a large batch takes the chunked route: create this device's copy
    // streams now, so that the first call can already be captured
    std::lock_guard<std::mutex> lock(g_pipe_mu);
    PipeRes* res = nullptr;
    const cudaError_t e = pipe_resources(&res);
    if (e != cudaSuccess) {
      note_cuda_error(e, "sda_build_decode_host_workspace_size");
      return SDA_ERR_CUDA;
    }
  }
  return SDA_OK;
}

sda_status sda_build_decode_host(const int32_t* state_slot, const int32_t* swa_len,
                                 const int32_t* swa_head, const int32_t* comp_indptr,
                                 const int32_t* comp_block, const int32_t* comp_slot,
                                 int64_t comp_total, int win, int k_per_block, int64_t swa_pages,
                                 int64_t capacity, const void* q, const void* unified_kv,
                                 const float* kv_scale, int64_t total_pages,
                                 const float* attn_sink, float softmax_scale, int N, int H, int D,
                                 void* out, int32_t* status, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  if (!status || !workspace) return SDA_ERR_INVALID_ARG;
  // everything checkable on the host is checked before the input gather is enqueued
  sda_status r0 = build_decode_scalars_ok(N, win, k_per_block, swa_pages, total_pages, capacity,
                                          comp_total, unified_kv, kv_scale, attn_sink, H, D);
  if (r0 != SDA_OK) return r0;
  const bool fp8 = kv_scale != nullptr;
  if (!aligned(workspace, 256)) return SDA_ERR_WORKSPACE;
  // every host array must be page-locked; q and out 16-byte aligned
  const void* d_st = host_view(status);
  const void* d_ss = N > 0 ? host_view(state_slot) : nullptr;
  const void* d_sl = N > 0 ? host_view(swa_len) : nullptr;
  const void* d_sh = N > 0 ? host_view(swa_head) : nullptr;
  const void* d_cp = host_view(comp_indptr);
  const void* d_cb = comp_total > 0 ? host_view(comp_block) : nullptr;
  const void* d_cs = comp_total > 0 ? host_view(comp_slot) : nullptr;
  const void* d_q = N > 0 ? host_view(q) : nullptr;
  const void* d_out = N > 0 ? host_view(out) : nullptr;
  if (!d_st || !d_cp || (N > 0 && (!d_ss || !d_sl || !d_sh || !d_q || !d_out)) ||
      (comp_total > 0 && (!d_cb || !d_cs)))
    return SDA_ERR_INVALID_ARG;
  if ((N > 0 && (!aligned(d_q, 16) || !aligned(d_out, 16))) || !aligned(d_st, 4) ||
      !aligned(d_cp, 4) || (N > 0 && (!aligned(d_ss, 4) || !aligned(d_sl, 4) || !aligned(d_sh, 4))) ||
      (comp_total > 0 && (!aligned(d_cb, 4) || !aligned(d_cs, 4))))
    return SDA_ERR_INVALID_ARG;
  size_t dec = 0;
  sda_status r = build_decode_ws(N, H, D, capacity, fp8, &dec);
  if (r != SDA_OK) return r;
  const HostWs w = host_ws_layout(N, H, D, comp_total, capacity, dec);
  if (workspace_bytes < w.total) return SDA_ERR_WORKSPACE;
  char* base = static_cast<char*>(workspace);
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if ((int64_t)N * H * D * 2 >= kPipelineBytes && N >= 2)
    return build_decode_host_pipelined(state_slot, swa_len, swa_head, comp_indptr, comp_block,
                                       comp_slot, comp_total, win, k_per_block, swa_pages, capacity,
                                       q, unified_kv, kv_scale, total_pages, attn_sink,
                                       softmax_scale, N, H, D, out, status, base, w, st);
  DeviceCaps caps;
  cudaError_t e = device_caps(&caps);
  const int64_t q_words = (int64_t)N * H * D / 2;
  CopySegments in = {};
  auto add = [](CopySegments& c, const void* src, void* dst, int64_t words) {
    if (words > 0) c.seg[c.n++] = CopySegment{src, dst, words};
  };
  add(in, d_q, base + w.q, q_words);
  add(in, d_ss, base + w.ss, N);
  add(in, d_sl, base + w.sl, N);
  add(in, d_sh, base + w.sh, N);
  add(in, d_cp, base + w.cptr, N + 1);
  add(in, d_cb, base + w.cb, comp_total);
  add(in, d_cs, base + w.cs, comp_total);
  if (e == cudaSuccess) e = launch_gather_copy(in, caps.num_sms, st);
  if (e != cudaSuccess) {
    note_cuda_error(e, "sda_build_decode_host");
    return SDA_ERR_CUDA;
  }
  r = build_decode_impl(reinterpret_cast<const int32_t*>(base + w.ss),
                        reinterpret_cast<const int32_t*>(base + w.sl),
                        reinterpret_cast<const int32_t*>(base + w.sh),
                        reinterpret_cast<const int32_t*>(base + w.cptr),
                        reinterpret_cast<const int32_t*>(base + w.cb),
                        reinterpret_cast<const int32_t*>(base + w.cs), comp_total, win,
                        k_per_block, swa_pages, reinterpret_cast<int32_t*>(base + w.idx), capacity,
                        reinterpret_cast<int32_t*>(base + w.iptr),
                        reinterpret_cast<int32_t*>(base + w.st), base + w.q, unified_kv, kv_scale,
                        total_pages, attn_sink, softmax_scale, N, H, D, base + w.out,
                        base + w.dec, dec > 0 ? dec : 1, stream, "sda_build_decode_host");
  if (r != SDA_OK) return r;
  CopySegments back = {};
  add(back, base + w.out, const_cast<void*>(d_out), q_words);
  add(back, base + w.st, const_cast<void*>(d_st), 1);
  e = launch_gather_copy(back, caps.num_sms, st);
  if (e != cudaSuccess) {
    note_cuda_error(e, "sda_build_decode_host");
    return SDA_ERR_CUDA;
  }
  return SDA_OK;
}

sda_status sda_decode_kernel(int H, int D, int* kernel) {
  if (!kernel) return SDA_ERR_INVALID_ARG;
  if (!shape_supported(H, D)) return SDA_ERR_UNSUPPORTED;
  DeviceCaps caps;
  cudaError_t e = device_caps(&caps);
  if (e != cudaSuccess) {
    note_cuda_error(e, "sda_decode_kernel");
    return SDA_ERR_CUDA;
  }
  LaunchPlan lp;
  choose_plan(H, D, caps, &lp);
  static_assert(SDA_KERNEL_SIMT == kSimt && SDA_KERNEL_ONE_CTA == kUmma, "public kernel codes");
  *kernel = lp.variant;
  return SDA_OK;
}

sda_status sda_debug_wait_fault(int withhold_arrive, uint64_t timeout_ns) {
  if (withhold_arrive != 0 && withhold_arrive != 1) return SDA_ERR_INVALID_ARG;
  g_withhold_arrive.store(withhold_arrive);
  g_wait_timeout_ns.store(timeout_ns);
  return SDA_OK;
}

sda_status sda_set_timing_events(void* before, void* after) {
  if ((before == nullptr) != (after == nullptr)) return SDA_ERR_INVALID_ARG;
  g_ev_before = static_cast<cudaEvent_t>(before);
  g_ev_after = static_cast<cudaEvent_t>(after);
  return SDA_OK;
}

sda_status sda_decode_error_flag(const void* workspace, int32_t* device_flag, void* stream) {
  if (!workspace || !device_flag || !aligned(workspace, 256)) return SDA_ERR_INVALID_ARG;
  const char* src = static_cast<const char*>(workspace) + offsetof(WsHeader, error);
  cudaError_t e = cudaMemcpyAsync(device_flag, src, sizeof(int32_t), cudaMemcpyDeviceToDevice,
                                  static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    note_cuda_error(e, "sda_decode_error_flag");
    return SDA_ERR_CUDA;
  }
  return SDA_OK;
}

sda_status sda_build_indices(const int32_t* state_slot, const int32_t* swa_len,
                             const int32_t* swa_head, const int32_t* comp_indptr,
                             const int32_t* comp_block, const int32_t* comp_slot,
                             int64_t comp_total, int N, int win, int k_per_block,
                             int64_t swa_pages, int64_t total_pages, int32_t* kv_indices,
                             int64_t capacity, int32_t* kv_indptr, int32_t* status,
                             void* stream) {
  if (N < 0 || win <= 0 || k_per_block <= 0 || swa_pages < 0 || total_pages <= 0 ||
      total_pages > 0x7fffffffll || swa_pages > total_pages || capacity < 0 ||
      capacity > 0x7fffffffll || comp_total < 0 || comp_total > 0x7fffffffll)
    return SDA_ERR_INVALID_ARG;
  if (!kv_indptr || !status) return SDA_ERR_INVALID_ARG;
  if (N > 0 && (!state_slot || !swa_len || !swa_head || !comp_indptr)) return SDA_ERR_INVALID_ARG;
  if (comp_total > 0 && (!comp_block || !comp_slot)) return SDA_ERR_INVALID_ARG;
  if (capacity > 0 && !kv_indices) return SDA_ERR_INVALID_ARG;
  cudaError_t e = launch_build_indices(state_slot, swa_len, swa_head, comp_indptr, comp_block,
                                       comp_slot, comp_total, N, win, k_per_block, swa_pages,
                                       total_pages, kv_indices, capacity, kv_indptr, status,
                                       static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    note_cuda_error(e, "sda_build_indices");
    return SDA_ERR_CUDA;
  }
  return SDA_OK;
}

sda_status sda_validate_indices(const int32_t* kv_indices, int64_t total_indices,
                                const int32_t* kv_indptr, int N, int64_t total_pages,
                                int32_t* status, void* stream) {
  if (N < 0 || total_indices < 0 || total_pages <= 0 || !kv_indptr || !status)
    return SDA_ERR_INVALID_ARG;
  if (total_indices > 0 && !kv_indices) return SDA_ERR_INVALID_ARG;
  cudaError_t e = launch_validate(kv_indices, total_indices, kv_indptr, N, total_pages, status,
                                  static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    note_cuda_error(e, "sda_validate_indices");
    return SDA_ERR_CUDA;
  }
  return SDA_OK;
}

sda_status sda_topk_slots(const float* scores, int64_t score_stride, const int32_t* lengths,
                          const int32_t* block_table, int64_t bt_stride, int N, int k,
                          int k_per_block, int32_t* comp_indptr, int32_t* comp_block,
                          int32_t* comp_slot, int64_t capacity, int32_t* status, void* stream) {
  if (N < 0 || k < 0 || k_per_block <= 0 || score_stride < 0 || score_stride > 0x7fffffffll ||
      bt_stride < 0 || bt_stride * static_cast<int64_t>(k_per_block) < score_stride ||
      capacity < 0 || capacity > 0x7fffffffll)
    return SDA_ERR_INVALID_ARG;
  if (!comp_indptr || !status) return SDA_ERR_INVALID_ARG;
  if (N > 0 && !lengths) return SDA_ERR_INVALID_ARG;
  if (N > 0 && k > 0 && score_stride > 0 && (!scores || !block_table)) return SDA_ERR_INVALID_ARG;
  if (capacity > 0 && (!comp_block || !comp_slot)) return SDA_ERR_INVALID_ARG;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(status, 0, sizeof(int32_t), st);
  if (e == cudaSuccess && g_ev_before && g_ev_after) e = cudaEventRecord(g_ev_before, st);
  if (e == cudaSuccess)
    e = launch_topk_slots(scores, score_stride, lengths, block_table, bt_stride, N, k,
                          k_per_block, comp_indptr, comp_block, comp_slot, capacity, status, st);
  if (e == cudaSuccess && g_ev_before && g_ev_after) e = cudaEventRecord(g_ev_after, st);
  if (e != cudaSuccess) {
    note_cuda_error(e, "sda_topk_slots");
    return SDA_ERR_CUDA;
  }
  return SDA_OK;
}

static sda_status store_common(const void* q, const void* kv, const void* q_norm_w,
                               const void* kv_norm_w, const float* cos_cache,
                               const float* sin_cache, int max_pos, const int32_t* positions,
                               const int32_t* state_slot, int N, int H, int D, int rope_dim,
                               float eps, int win, int64_t swa_pages, int64_t total_pages,
                               void* q_out, void* pool, uint8_t* pool_fp8, float* pool_scale,
                               int32_t* status, void* stream, const char* who) {
  using namespace sda;
  if (N < 0 || H < 1 || D < 8 || D > 2048 || D % 8 || rope_dim < 0 || rope_dim > D ||
      rope_dim % 8 || max_pos < 0 || win <= 0 || swa_pages < 0 || total_pages <= 0 ||
      swa_pages > total_pages || !(eps >= 0.f) || !std::isfinite(eps))
    return SDA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(N) * (H + 1) > (int64_t{1} << 30)) return SDA_ERR_INVALID_ARG;
  if (!status || !q_norm_w || !kv_norm_w) return SDA_ERR_INVALID_ARG;
  if (N > 0 && (!q || !kv || !positions || !state_slot || !q_out)) return SDA_ERR_INVALID_ARG;
  if (N > 0 && rope_dim > 0 && max_pos > 0 && (!cos_cache || !sin_cache)) return SDA_ERR_INVALID_ARG;
  if (N > 0 && !pool && !pool_fp8) return SDA_ERR_INVALID_ARG;
  if (pool_fp8 && !pool_scale) return SDA_ERR_INVALID_ARG;
  const void* vec16[] = {q, kv, q_norm_w, kv_norm_w, q_out, pool, pool_fp8, cos_cache, sin_cache};
  for (const void* ptr : vec16)
    if (ptr && !aligned(ptr, 16)) return SDA_ERR_INVALID_ARG;
  if (pool_scale && !aligned(pool_scale, 4)) return SDA_ERR_INVALID_ARG;
  // q_out is either q itself (in place) or a disjoint buffer.
  const size_t qbytes = (size_t)N * H * D * 2;
  const uintptr_t a = reinterpret_cast<uintptr_t>(q), b = reinterpret_cast<uintptr_t>(q_out);
  if (N > 0 && a != b && a < b + qbytes && b < a + qbytes) return SDA_ERR_INVALID_ARG;
  DeviceCaps caps;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = device_caps(&caps);
  if (e == cudaSuccess) e = cudaMemsetAsync(status, 0, sizeof(int32_t), st);
  if (e == cudaSuccess && g_ev_before && g_ev_after) e = cudaEventRecord(g_ev_before, st);
  if (e == cudaSuccess)
    e = launch_qk_norm_rope_store(q, kv, q_norm_w, kv_norm_w, cos_cache, sin_cache, max_pos,
                                  positions, state_slot, N, H, D, rope_dim, eps, win, swa_pages,
                                  q_out, pool, pool_fp8, pool_scale, status, caps.num_sms, st);
  if (e == cudaSuccess && g_ev_before && g_ev_after) e = cudaEventRecord(g_ev_after, st);
  if (e != cudaSuccess) {
    note_cuda_error(e, who);
    return SDA_ERR_CUDA;
  }
  return SDA_OK;
}

sda_status sda_qk_norm_rope_swa_store(const void* q, const void* kv, const void* q_norm_w,
                                      const void* kv_norm_w, const float* cos_cache,
                                      const float* sin_cache, int max_pos,
                                      const int32_t* positions, const int32_t* state_slot, int N,
                                      int H, int D, int rope_dim, float eps, int win,
                                      int64_t swa_pages, int64_t total_pages, void* q_out,
                                      void* unified_kv, int32_t* status, void* stream) {
  if (N > 0 && !unified_kv) return SDA_ERR_INVALID_ARG;
  return store_common(q, kv, q_norm_w, kv_norm_w, cos_cache, sin_cache, max_pos, positions,
                      state_slot, N, H, D, rope_dim, eps, win, swa_pages, total_pages, q_out,
                      unified_kv, nullptr, nullptr, status, stream, "sda_qk_norm_rope_swa_store");
}

sda_status sda_qk_norm_rope_swa_store_fp8(const void* q, const void* kv, const void* q_norm_w,
                                          const void* kv_norm_w, const float* cos_cache,
                                          const float* sin_cache, int max_pos,
                                          const int32_t* positions, const int32_t* state_slot,
                                          int N, int H, int D, int rope_dim, float eps, int win,
                                          int64_t swa_pages, int64_t total_pages, void* q_out,
                                          void* kv_fp8, float* kv_scale, int32_t* status,
                                          void* stream) {
  if (N > 0 && (!kv_fp8 || !kv_scale)) return SDA_ERR_INVALID_ARG;
  return store_common(q, kv, q_norm_w, kv_norm_w, cos_cache, sin_cache, max_pos, positions,
                      state_slot, N, H, D, rope_dim, eps, win, swa_pages, total_pages, q_out,
                      nullptr, static_cast<uint8_t*>(kv_fp8), kv_scale, status, stream,
                      "sda_qk_norm_rope_swa_store_fp8");
}

}  // extern "C"
