// sda_decode_umma.cu -- tensor-core (tcgen05 / TMEM / TMA) decode kernel for
// D = 512 and H a multiple of 16 (16, 32, 64, or multiples of 64).
//
// What it computes is the paged_decode.py docstring quoted on the sglang
// PR 28392 summary page ("关键源码片段": caller convention, returns,
// numerics): for each token t and head h, attention of q[t,h] over the rows
// unified_kv[kv_indices[kv_indptr[t]:kv_indptr[t+1]]] -- each row is both key
// and value -- with the per-head sink as a virtual key of zero value, an
// fp32 online softmax in the log2 domain (qk_scale = softmax_scale * log2 e),
// out in bf16.
//
// Design for GB300 (not from the page, whose kernel targets AMD GPUs):
//  * One persistent CTA per SM owns one work unit at a time: a piece of one
//    token's slot list for NH <= 64 heads (H = 128 uses two CTAs per token).
//    All heads of a token share each gathered KV row, so a row is read from
//    HBM once per CTA.
//  * Warp 0 gathers KV tiles of 64 slots with TMA tile::gather4 (four rows x
//    128 bytes per instruction) into 128-byte-swizzled shared memory, two
//    stages deep, and loads q[t] with plain tiled TMA.
//  * Warp 1 issues tcgen05 MMAs:  S = Q K^T  (M = 64 padded heads, N = 64
//    slots, K = 512) into TMEM, then  O^T += V^T P^T  (M = 128 rows of D,
//    N = NH heads, K = 64 slots) into a TMEM accumulator.  The same shared
//    tile is K (K-major operand) and V (MN-major operand).
//  * Warps 2..5 read S rows from TMEM (one head per thread), run the online
//    softmax, write P (bf16) to shared memory, rescale O^T in TMEM only when
//    a head's running max grows by more than 8 (2^8 headroom, so p <= 256),
//    and finally normalise with the sink and write out (or, for a piece of a
//    split token, write the unnormalised partial for the combine kernel).
//  * Every mbarrier wait is bounded (2 s); on timeout the kernel raises the
//    workspace error word, drains its own copies and returns.
#include <cuda.h>
#include <cuda_bf16.h>

#include "sda_internal.cuh"
#include "umma_ptx.cuh"

namespace sda {

namespace {

using namespace ptx;

constexpr int kD = 512;
constexpr int kPanels = kD / 64;           // 128-byte column panels per row
constexpr int kTileN = kTileSlots;         // 64 slots per KV tile
constexpr int kQRows = 64;                 // QK MMA M (heads padded to 64)
constexpr int kPanelQ = kQRows * 128;      // bytes of one Q panel
constexpr int kPanelKV = kTileN * 128;     // bytes of one KV panel
constexpr int kQBytes = kPanels * kPanelQ;     // 64 KB
constexpr int kKVBytes = kPanels * kPanelKV;   // 64 KB per stage
constexpr int kStages = 2;
constexpr int kThreads = 192;              // 6 warps
constexpr int kSoftmaxWarp0 = 2;           // warps 2..5: softmax / epilogue
constexpr int kSoftmaxThreads = 128;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;

enum Bar : int {
  kBarQFull = 0,
  kBarQEmpty,
  kBarKVFull0,
  kBarKVFull1,
  kBarPVDone0,
  kBarPVDone1,
  kBarSFull0,
  kBarSFull1,
  kBarSEmpty0,
  kBarSEmpty1,
  kBarPFull0,
  kBarPFull1,
  kBarOEmpty,
  kBarDrain,
  kNumBars
};

template <int NH>
struct Cfg {
  static constexpr int kPBytes = NH * 128;  // P: NH rows x 64 slots bf16
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = kQBytes;
  static constexpr int kOffP = kOffKV + kStages * kKVBytes;
  static constexpr int kOffBar = kOffP + kStages * kPBytes;
  static constexpr int kOffMisc = kOffBar + 128;
  // misc: tmem base (4), abort flag (4), pad, then per-head float arrays
  static constexpr int kOffAlpha = kOffMisc + 16;
  static constexpr int kOffFac = kOffAlpha + 4 * 64;
  static constexpr int kSmemUsed = kOffFac + 4 * 64;
  static constexpr int kSmem = kSmemUsed + 1024;  // slack for 1024-byte alignment
  static constexpr int kTmemCols = (128 + 4 * NH) <= 256 ? 256 : 512;
  static constexpr int kOCol = 128;  // O^T block b at columns [128 + b*NH, +NH)
  static constexpr uint32_t kIdescQK = idesc_bf16_f32(64, 64, false, false);
  static constexpr uint32_t kIdescPV = idesc_bf16_f32(128, NH, true, false);
  static_assert(kOffP % 1024 == 0 && kPBytes % 1024 == 0, "swizzle atoms need 1 KB alignment");
  static_assert(kSmem <= 232448, "shared memory budget");
};

struct Params {
  const __nv_bfloat16* q;
  const int32_t* kv_indices;
  const float* attn_sink;
  __nv_bfloat16* out;
  WsHeader* hdr;
  const int4* units;
  float2* part_ml;
  float* part_o;
  float qk_scale_log2;
  int H;
};

// Bounded wait.  Returns false (and raises the abort flags) on timeout; once
// any role has aborted, every later wait returns false at once, so all roles
// run to the end of their loops quickly and the CTA exits.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         WsHeader* hdr) {
  if (mbar_try_wait(bar, parity)) return true;
  if (*abort_flag) return false;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > kWaitTimeoutNs) {
        *abort_flag = 1;
        atomicExch(&hdr->error, 1);
        return false;
      }
    }
  }
}

// Wait used only while draining copies / MMAs this CTA started: bounded by
// the timeout, but not cut short by the abort flag.
__device__ __forceinline__ void drain_bar(uint32_t bar, uint32_t parity, WsHeader* hdr) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kWaitTimeoutNs) {
      atomicExch(&hdr->error, 1);
      return;
    }
  }
}

template <int NH>
__global__ void __launch_bounds__(kThreads, 1)
decode_umma_kernel(const __grid_constant__ CUtensorMap tmap_q,
                   const __grid_constant__ CUtensorMap tmap_kv, const Params p) {
  using C = Cfg<NH>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_addr(smem);
  const uint32_t sQ = sbase + C::kOffQ;
  const uint32_t sKV = sbase + C::kOffKV;
  const uint32_t sP = sbase + C::kOffP;
  const uint32_t sBar = sbase + C::kOffBar;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
  float* s_alpha = reinterpret_cast<float*>(smem + C::kOffAlpha);
  float* s_fac = reinterpret_cast<float*>(smem + C::kOffFac);
  auto bar = [&](int i) { return sBar + 8u * (uint32_t)i; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(bar(kBarQFull), 1);
    mbar_init(bar(kBarQEmpty), 1);
    mbar_init(bar(kBarKVFull0), 1);
    mbar_init(bar(kBarKVFull1), 1);
    mbar_init(bar(kBarPVDone0), 1);
    mbar_init(bar(kBarPVDone1), 1);
    mbar_init(bar(kBarSFull0), 1);
    mbar_init(bar(kBarSFull1), 1);
    mbar_init(bar(kBarSEmpty0), 4);
    mbar_init(bar(kBarSEmpty1), 4);
    mbar_init(bar(kBarPFull0), 4);
    mbar_init(bar(kBarPFull1), 4);
    mbar_init(bar(kBarOEmpty), 4);
    mbar_init(bar(kBarDrain), 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmap_q);
    tma_prefetch_desc(&tmap_kv);
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int n_units = p.hdr->n_units;
  const int H = p.H;

  if (warp == 0) {
    // ===================================================== TMA producer
    int g = 0, nu = 0, q_issued = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int pos = unit_position(k, blockIdx.x, gridDim.x);
      if (pos >= n_units) break;
      const int4 u = p.units[pos];
      const int len = u.z;
      if (len <= 0) continue;
      const int hg = unit_head_group(u.w);
      const int ntiles = (len + kTileN - 1) / kTileN;
      if (lane == 0) {
        if (nu >= 1) ok = wait_bar(bar(kBarQEmpty), (nu - 1) & 1, abort_flag, p.hdr);
        if (ok) {
          mbar_arrive_expect_tx(bar(kBarQFull), NH * 128 * kPanels);
          const int qrow = u.x * H + hg * NH;
#pragma unroll
          for (int c = 0; c < kPanels; ++c) tma_load_2d(sQ + c * kPanelQ, &tmap_q, c * 64, qrow, bar(kBarQFull));
          q_issued = nu + 1;
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      for (int i = 0; i < ntiles && ok; ++i, ++g) {
        const int s = g & 1;
        const int base = u.y + i * kTileN;
        const int n = min(kTileN, len - i * kTileN);
        int i0 = lane < n ? __ldg(p.kv_indices + base + lane) : 0;
        int i1 = lane + 32 < n ? __ldg(p.kv_indices + base + lane + 32) : 0;
        const int first = __shfl_sync(0xffffffffu, i0, 0);
        if (lane >= n) i0 = first;        // pad the tail with a valid row;
        if (lane + 32 >= n) i1 = first;   // its probability is forced to 0
        if (lane == 0 && g >= 2) ok = wait_bar(bar(kBarPVDone0 + s), ((g >> 1) - 1) & 1, abort_flag, p.hdr);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        if (lane == 0) mbar_arrive_expect_tx(bar(kBarKVFull0 + s), kKVBytes);
        __syncwarp();
        const int g4 = lane & 15;
        int y[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int row = 4 * g4 + r;
          const int a = __shfl_sync(0xffffffffu, i0, row & 31);
          const int b = __shfl_sync(0xffffffffu, i1, row & 31);
          y[r] = row < 32 ? a : b;
        }
        const uint32_t dst0 = sKV + s * kKVBytes + g4 * 512;
        const int c0 = (lane >> 4) * 4;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const int c = c0 + cc;
          tma_gather4(dst0 + c * kPanelKV, &tmap_kv, c * 64, y[0], y[1], y[2], y[3], bar(kBarKVFull0 + s));
        }
      }
      ++nu;
    }
    // drain: make sure every copy this warp started has landed before exit
    if (lane == 0) {
      for (int gg = (g >= 2 ? g - 2 : 0); gg < g; ++gg)
        drain_bar(bar(kBarKVFull0 + (gg & 1)), (gg >> 1) & 1, p.hdr);
      if (q_issued >= 1) drain_bar(bar(kBarQFull), (q_issued - 1) & 1, p.hdr);
    }
  } else if (warp == 1) {
    // ===================================================== MMA issuer
    if (lane == 0) {
      int g = 0, nu = 0;
      bool ok = true;
      auto issue_pv = [&](int gp, bool first, int nu_cur) -> bool {
        const int sp = gp & 1;
        if (!wait_bar(bar(kBarPFull0 + sp), (gp >> 1) & 1, abort_flag, p.hdr)) return false;
        if (first && nu_cur >= 1)
          if (!wait_bar(bar(kBarOEmpty), (nu_cur - 1) & 1, abort_flag, p.hdr)) return false;
        tc_fence_after();
        const uint32_t kvs = sKV + sp * kKVBytes;
        const uint32_t ps = sP + sp * C::kPBytes;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            // A = V^T block b: rows d in [128b, 128b+128) = panels 2b, 2b+1 (MN-major);
            //     K = slots [16kk, 16kk+16) = row groups 2kk, 2kk+1
            const uint64_t a = sdesc_sw128(kvs + (2 * b) * kPanelKV + kk * 2048, kPanelKV, 1024);
            // B = P^T: N = NH heads (rows), K = 16 slots at byte offset 32kk (K-major)
            const uint64_t bd = sdesc_sw128(ps + kk * 32, 16, 1024);
            mma_bf16(tmem + C::kOCol + b * NH, a, bd, C::kIdescPV, (first && kk == 0) ? 0u : 1u);
          }
        }
        mma_commit(bar(kBarPVDone0 + sp));
        return true;
      };
      for (int k = 0; ok; ++k) {
        const int pos = unit_position(k, blockIdx.x, gridDim.x);
        if (pos >= n_units) break;
        const int4 u = p.units[pos];
        const int len = u.z;
        if (len <= 0) continue;
        const int ntiles = (len + kTileN - 1) / kTileN;
        ok = wait_bar(bar(kBarQFull), nu & 1, abort_flag, p.hdr);
        for (int i = 0; i < ntiles && ok; ++i, ++g) {
          const int s = g & 1;
          ok = wait_bar(bar(kBarKVFull0 + s), (g >> 1) & 1, abort_flag, p.hdr);
          if (ok && g >= 2) ok = wait_bar(bar(kBarSEmpty0 + s), ((g >> 1) - 1) & 1, abort_flag, p.hdr);
          if (!ok) break;
          tc_fence_after();
          const uint32_t kvs = sKV + s * kKVBytes;
#pragma unroll
          for (int c = 0; c < kPanels; ++c) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t a = sdesc_sw128(sQ + c * kPanelQ + kk * 32, 16, 1024);
              const uint64_t bd = sdesc_sw128(kvs + c * kPanelKV + kk * 32, 16, 1024);
              mma_bf16(tmem + s * 64, a, bd, C::kIdescQK, (c | kk) ? 1u : 0u);
            }
          }
          mma_commit(bar(kBarSFull0 + s));
          if (i == ntiles - 1) mma_commit(bar(kBarQEmpty));
          if (i >= 1) ok = issue_pv(g - 1, i == 1, nu);
        }
        if (ok) ok = issue_pv(g - 1, ntiles == 1, nu);
        ++nu;
      }
      // drain the tensor pipe before TMEM is released
      mma_commit(bar(kBarDrain));
      drain_bar(bar(kBarDrain), 0, p.hdr);
    }
    __syncwarp();
  } else {
    // ===================================================== softmax + epilogue
    const int q4 = warp & 3;                  // TMEM lane quadrant of this warp
    const int st = threadIdx.x - kSoftmaxWarp0 * 32;  // 0..127
    // M = 64 accumulator layout: row r lives in lane 32*(r/16) + r%16.
    const int head = (lane < 16) ? q4 * 16 + lane : -1;
    const bool has_head = head >= 0 && head < NH;
    const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
    // Control flow here is identical in the four warps (it depends only on
    // the unit list and on block-wide votes), so every named barrier is
    // reached by all 128 threads even after a wait timed out: a timed-out
    // wait only leaves garbage in the outputs and the error word raised.
    int g = 0;
    for (int k = 0;; ++k) {
      const int pos = unit_position(k, blockIdx.x, gridDim.x);
      if (pos >= n_units) break;
      const int4 u = p.units[pos];
      const int t = u.x, len = u.z, hg = unit_head_group(u.w), row = unit_part_row(u.w);
      if (len <= 0) {
        // padded token: out = 0 for its NH heads (contiguous NH*D bf16)
        uint4* o = reinterpret_cast<uint4*>(p.out + ((size_t)t * H + hg * NH) * kD);
        for (int e = st; e < NH * kD / 8; e += kSoftmaxThreads) o[e] = make_uint4(0, 0, 0, 0);
        continue;
      }
      const int ntiles = (len + kTileN - 1) / kTileN;
      float m = -INFINITY, l = 0.f;
      for (int i = 0; i < ntiles; ++i, ++g) {
        const int s = g & 1;
        wait_bar(bar(kBarSFull0 + s), (g >> 1) & 1, abort_flag, p.hdr);
        tc_fence_after();
        uint32_t sv[64];
#pragma unroll
        for (int c = 0; c < 4; ++c)
          tmem_ld16(tmem + lane_base + s * 64 + c * 16, *reinterpret_cast<uint32_t(*)[16]>(sv + 16 * c));
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarSEmpty0 + s));
        const int n = min(kTileN, len - i * kTileN);
        float alpha = 1.f;
        bool need_rescale = false;
        uint32_t pk[32];
        if (has_head) {
          float y[64];
          float tmax = -INFINITY;
#pragma unroll
          for (int j = 0; j < 64; ++j) {
            y[j] = j < n ? __uint_as_float(sv[j]) * p.qk_scale_log2 : -INFINITY;
            tmax = fmaxf(tmax, y[j]);
          }
          if (tmax > m + kRescaleThreshold) {
            alpha = ex2_approx(m - tmax);  // 0 on the first tile (m = -inf)
            need_rescale = i > 0;
            l *= alpha;
            m = tmax;
          }
          float ls = 0.f;
#pragma unroll
          for (int j = 0; j < 64; j += 2) {
            const float p0 = ex2_approx(y[j] - m), p1 = ex2_approx(y[j + 1] - m);
            ls += p0 + p1;
            __nv_bfloat162 b2 = __floats2bfloat162_rn(p0, p1);
            pk[j >> 1] = *reinterpret_cast<uint32_t*>(&b2);
          }
          l += ls;
        }
        // P buffer s is free once the PV of tile g-2 is done
        if (g >= 2) {
          if (lane == 0) wait_bar(bar(kBarPVDone0 + s), ((g >> 1) - 1) & 1, abort_flag, p.hdr);
          __syncwarp();
        }
        if (has_head) {
          // row `head` of P (K-major, 128-byte swizzle): chunk c at (c ^ (head & 7)) * 16
          uint8_t* prow = smem + C::kOffP + s * C::kPBytes + (head >> 3) * 1024 + (head & 7) * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4*>(prow + ((c ^ (head & 7)) << 4)) =
                make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
        }
        fence_proxy_async_smem();
        if (named_bar_or(1, kSoftmaxThreads, need_rescale)) {
          if (has_head) s_alpha[head] = alpha;
          named_bar_sync(1, kSoftmaxThreads);
          // O^T must be quiescent: wait for the PV of tile g-1
          if (lane == 0) wait_bar(bar(kBarPVDone0 + ((g - 1) & 1)), ((g - 1) >> 1) & 1, abort_flag, p.hdr);
          __syncwarp();
          tc_fence_after();
#pragma unroll
          for (int b = 0; b < 4; ++b) {
#pragma unroll
            for (int c = 0; c < NH / 16; ++c) {
              uint32_t ov[16];
              const uint32_t ta = tmem + lane_base + C::kOCol + b * NH + c * 16;
              tmem_ld16(ta, ov);
              tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 16; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * s_alpha[c * 16 + e]);
              tmem_st16(ta, ov);
            }
          }
          tmem_wait_st();
          named_bar_sync(1, kSoftmaxThreads);  // s_alpha is rewritten next time
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarPFull0 + s));
      }
      // ---------------------------------------------- epilogue of the unit
      const int gl = g - 1;
      if (lane == 0) wait_bar(bar(kBarPVDone0 + (gl & 1)), (gl >> 1) & 1, abort_flag, p.hdr);
      __syncwarp();
      tc_fence_after();
      if (has_head) {
        const int hh = hg * NH + head;
        if (row < 0) {
          const float ms = p.attn_sink[hh] * kLog2e;
          const float M = fmaxf(m, ms);
          float f = 0.f;
          if (M != -INFINITY && ms != INFINITY) {
            const float a = ex2_approx(m - M);
            f = a / (l * a + ex2_approx(ms - M));
          }
          s_fac[head] = f;
        } else {
          p.part_ml[(size_t)row * H + hh] = make_float2(m, l);
          s_fac[head] = 1.f;
        }
      }
      named_bar_sync(1, kSoftmaxThreads);
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int d = b * 128 + q4 * 32 + lane;
#pragma unroll
        for (int c = 0; c < NH / 16; ++c) {
          uint32_t ov[16];
          tmem_ld16(tmem + lane_base + C::kOCol + b * NH + c * 16, ov);
          tmem_wait_ld();
          if (row < 0) {
            __nv_bfloat16* o = p.out + ((size_t)t * H + hg * NH + c * 16) * kD + d;
#pragma unroll
            // "+ 0.f" turns -0 into +0 when the factor is 0 (sink = +inf)
            for (int e = 0; e < 16; ++e) o[(size_t)e * kD] = __float2bfloat16_rn(__uint_as_float(ov[e]) * s_fac[c * 16 + e] + 0.f);
          } else {
            float* o = p.part_o + ((size_t)row * H + hg * NH + c * 16) * kD + d;
#pragma unroll
            for (int e = 0; e < 16; ++e) o[(size_t)e * kD] = __uint_as_float(ov[e]);
          }
        }
      }
      tc_fence_before();
      named_bar_sync(1, kSoftmaxThreads);  // s_fac is rewritten by the next unit
      if (lane == 0) mbar_arrive(bar(kBarOEmpty));
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, C::kTmemCols);
}

// ------------------------------------------------------------------ host side
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  return fn;
}

bool make_map_2d(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint32_t box_cols,
                 uint32_t box_rows, CUtensorMapL2promotion promo) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, promo,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int NH>
cudaError_t launch_nh(const void* q, const void* kv, int64_t total_pages, const int32_t* kv_indices,
                      const float* attn_sink, float scale, int N, int H, void* out, void* ws,
                      const WsLayout& L, const LaunchPlan& lp, cudaStream_t st) {
  CUtensorMap tq, tkv;
  if (!make_map_2d(&tq, q, kD, (uint64_t)N * H, 64, NH, CU_TENSOR_MAP_L2_PROMOTION_L2_128B) ||
      !make_map_2d(&tkv, kv, kD, (uint64_t)total_pages, 64, 1, CU_TENSOR_MAP_L2_PROMOTION_L2_128B))
    return cudaErrorInvalidValue;
  char* base = static_cast<char*>(ws);
  Params p;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.kv_indices = kv_indices;
  p.attn_sink = attn_sink;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.hdr = reinterpret_cast<WsHeader*>(base);
  p.units = reinterpret_cast<const int4*>(base + L.units_off);
  p.part_ml = reinterpret_cast<float2*>(base + L.ml_off);
  p.part_o = reinterpret_cast<float*>(base + L.o_off);
  p.qk_scale_log2 = scale * kLog2e;
  p.H = H;
  decode_umma_kernel<NH><<<lp.grid, kThreads, Cfg<NH>::kSmem, st>>>(tq, tkv, p);
  return cudaGetLastError();
}

}  // namespace

size_t umma_smem_bytes(int nh) {
  switch (nh) {
    case 16: return Cfg<16>::kSmem;
    case 32: return Cfg<32>::kSmem;
    case 64: return Cfg<64>::kSmem;
    default: return 0;
  }
}

cudaError_t umma_prepare(int nh) {
  switch (nh) {
    case 16: return cudaFuncSetAttribute(decode_umma_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<16>::kSmem);
    case 32: return cudaFuncSetAttribute(decode_umma_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<32>::kSmem);
    case 64: return cudaFuncSetAttribute(decode_umma_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<64>::kSmem);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode_umma(const void* q, const void* kv, int64_t total_pages,
                               const int32_t* kv_indices, const float* attn_sink,
                               float softmax_scale, int N, int H, int D, void* out, void* ws,
                               const WsLayout& L, const LaunchPlan& lp, cudaStream_t st) {
  if (D != kD) return cudaErrorInvalidValue;
  switch (lp.nh) {
    case 16: return launch_nh<16>(q, kv, total_pages, kv_indices, attn_sink, softmax_scale, N, H, out, ws, L, lp, st);
    case 32: return launch_nh<32>(q, kv, total_pages, kv_indices, attn_sink, softmax_scale, N, H, out, ws, L, lp, st);
    case 64: return launch_nh<64>(q, kv, total_pages, kv_indices, attn_sink, softmax_scale, N, H, out, ws, L, lp, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace sda
