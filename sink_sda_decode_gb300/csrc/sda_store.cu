// sda_store.cu -- the step that fills the unified pool before decode: the
// per-head RMSNorm of q, the RMSNorm of the step's new KV row, GPT-J RoPE on
// the last R dims of both, and the store of the KV row into its SWA ring slot
// state_slot * win + pos mod win, as bf16 or as E4M3 codes with a
// power-of-two row scale.
//
// Source: the sglang PR 25898 summary page ("修复 DSV4 在 AMD GPU 上的运行时崩溃与
// JIT 不兼容"): section "关键文件" describes fused_qk_norm_rope_store.py as one
// kernel doing Q per-head RMSNorm, KV RMSNorm, RoPE, FP8 quantisation and the
// paged SWA store; section "关键符号" names _batched_rmsnorm, _gptj_rotate
// (adjacent-pair rotation) and fused_qk_norm_rope_swa_store; "实现拆解" item 2
// names the cos_cache / sin_cache.  The ring slot formula is the one of the
// paged_decode.py docstring on the PR 28392 page.  Power-of-two scales follow
// the UE8M0 scale rounding of the MXFP8 epilogue on the sglang attention tag
// page ("DSV4.1" entries).
//
// Layout of the work: rows are q[t, 0..H-1, :] and kv[t, :] (H + 1 rows of D
// elements per token, row H being the KV row).  One warp owns a row; lane l
// holds 16-byte chunks l, l + 32, ... (8 elements each), so every load and
// store of a row is one coalesced 512-byte access per chunk step and a RoPE
// pair (2i, 2i+1) never leaves its lane.  A warp keeps two rows' loads in
// flight.  The op is bound by HBM: each q element is read and written once
// (2 + 2 bytes), each KV element read once and written once to the pool.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "sda_internal.cuh"

namespace sda {

namespace {

constexpr int kStoreThreads = 256;

struct StoreParams {
  const uint16_t* q;          // [N, H, D] bf16
  const uint16_t* kv;         // [N, D] bf16
  const uint16_t* q_norm_w;   // [D] bf16
  const uint16_t* kv_norm_w;  // [D] bf16
  const float* cos_cache;     // [max_pos, R/2]
  const float* sin_cache;     // [max_pos, R/2]
  const int32_t* positions;   // [N]
  const int32_t* state_slot;  // [N]
  uint16_t* q_out;            // [N, H, D] bf16 (may be q itself)
  uint16_t* pool;             // bf16 pool [total_pages, D]          (bf16 store)
  uint8_t* pool_fp8;          // E4M3 codes [total_pages, D]         (FP8 store)
  float* pool_scale;          // [total_pages]                       (FP8 store)
  int32_t* status;
  int64_t rows;               // N * (H + 1)
  int64_t swa_pages;
  int N, H, D, R, max_pos, win;
  float eps;
};

__device__ __forceinline__ void unpack8(const uint4& v, float f[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    f[2 * k] = __uint_as_float(w[k] << 16);
    f[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
  }
}

// Packed fp32 pairs (Blackwell's f32x2 FMA pipe): one instruction, two IEEE
// round-to-nearest results, bit-identical to two scalar operations.
__device__ __forceinline__ uint64_t f2_pack(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}

__device__ __forceinline__ uint4 pack8_bf16(const float f[8]) {
  uint32_t w[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * k], f[2 * k + 1]);  // .x = low half
    w[k] = *reinterpret_cast<const uint32_t*>(&h);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// Eight values (already divided by the row scale) to eight E4M3 codes,
// rounded to nearest even and saturated to +-448; element 0 in the low byte.
__device__ __forceinline__ uint2 pack8_e4m3(const float f[8]) {
  uint32_t w[2] = {0u, 0u};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const __nv_fp8x2_storage_t two =
        __nv_cvt_float2_to_fp8x2(make_float2(f[2 * k], f[2 * k + 1]), __NV_SATFINITE, __NV_E4M3);
    w[k >> 1] |= static_cast<uint32_t>(two) << (16 * (k & 1));
  }
  return make_uint2(w[0], w[1]);
}

// e of the row scale 2^e: the least integer with 448 * 2^e >= amax, at least
// -126 (a normal fp32); 0 for amax = 0.  With amax = m * 2^E, m in [0.5, 1)
// and 448 = 0.875 * 2^9, the condition is 0.875 * 2^(9+e) >= m * 2^E: e = E - 9
// when m <= 0.875, else E - 8.  frexpf is exact, so is the result.
__device__ __forceinline__ int fp8_scale_exponent(float amax) {
  if (!(amax > 0.f)) return 0;
  int E;
  const float m = frexpf(amax, &E);
  const int e = (m <= 0.875f) ? E - 9 : E - 8;
  return e < -126 ? -126 : e;
}

// Norm, rotation, rounding and store of one loaded row x of token t (row
// `head` of it; head == H is the KV row).  With LASTJ the caller has already
// loaded this lane's RoPE factors of chunk CPL-1 (cs, sn): the rotated dims
// then all lie in that chunk (D a multiple of 256, R <= 256).  Otherwise they
// are loaded here.
template <int CPL, bool FP8, bool LASTJ>
__device__ __forceinline__ void process_row(const StoreParams& p, int lane, const uint4 (&x)[CPL],
                                            int t, int head, int st, int pos, float4 cs_last,
                                            float4 sn_last) {
  const int chunks = p.D >> 3;  // 16-byte chunks per row
  const int rope_chunk0 = (p.D - p.R) >> 3;
  const int half = p.R >> 1;
  const bool is_kv = head == p.H;
  const bool live = st >= 0 && pos >= 0 && pos < p.max_pos;
  if (!live) {
    if (!is_kv) {
      uint4* dst = reinterpret_cast<uint4*>(p.q_out + (static_cast<size_t>(t) * p.H + head) * p.D);
#pragma unroll
      for (int j = 0; j < CPL; ++j)
        if (lane + 32 * j < chunks) __stcs(dst + lane + 32 * j, make_uint4(0, 0, 0, 0));
    } else if (st >= 0 && lane == 0) {
      atomicOr(p.status, 1);  // a real token whose position has no cache row
    }
    return;
  }
  // RMSNorm: one sum of squares over the row (lane partials, then the warp).
  float f[CPL][8];
  uint64_t ss2 = 0;  // (even, odd) partial sums
#pragma unroll
  for (int j = 0; j < CPL; ++j) {
    unpack8(x[j], f[j]);
#pragma unroll
    for (int k = 0; k < 8; k += 2) {
      const uint64_t v = f2_pack(f[j][k], f[j][k + 1]);
      ss2 = f2_fma(v, v, ss2);
    }
  }
  float ss_even, ss_odd;
  f2_unpack(ss2, ss_even, ss_odd);
  float ss = ss_even + ss_odd;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  const float inv_rms = 1.0f / sqrtf(ss / static_cast<float>(p.D) + p.eps);
  float amax = 0.f;
  const uint4* wrow = reinterpret_cast<const uint4*>(is_kv ? p.kv_norm_w : p.q_norm_w);
#pragma unroll
  for (int j = 0; j < CPL; ++j) {
    const int c = lane + 32 * j;
    float w[8];
    unpack8(c < chunks ? __ldg(wrow + c) : make_uint4(0, 0, 0, 0), w);  // L1-resident
    const uint64_t inv2 = f2_pack(inv_rms, inv_rms);
#pragma unroll
    for (int k = 0; k < 8; k += 2) {  // (x * r) * w, as two scalar products would round
      const uint64_t y = f2_mul(f2_mul(f2_pack(f[j][k], f[j][k + 1]), inv2),
                                f2_pack(w[k], w[k + 1]));
      f2_unpack(y, f[j][k], f[j][k + 1]);
    }
    if (c >= rope_chunk0 && c < chunks && (!LASTJ || j == CPL - 1)) {
      // GPT-J rotation of the pairs (2i, 2i+1), i = 4 (c - rope_chunk0) + 0..3.
      float4 cs = cs_last, sn = sn_last;
      if (!LASTJ) {
        const size_t off = static_cast<size_t>(pos) * half + 4 * (c - rope_chunk0);
        cs = __ldg(reinterpret_cast<const float4*>(p.cos_cache + off));
        sn = __ldg(reinterpret_cast<const float4*>(p.sin_cache + off));
      }
      const float cv[4] = {cs.x, cs.y, cs.z, cs.w}, sv[4] = {sn.x, sn.y, sn.z, sn.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float a = f[j][2 * i], b = f[j][2 * i + 1];
        f[j][2 * i] = a * cv[i] - b * sv[i];
        f[j][2 * i + 1] = b * cv[i] + a * sv[i];
      }
    }
    if (FP8 && is_kv && c < chunks) {
#pragma unroll
      for (int k = 0; k < 8; ++k) amax = fmaxf(amax, fabsf(f[j][k]));
    }
  }
  if (!is_kv) {
    uint4* dst = reinterpret_cast<uint4*>(p.q_out + (static_cast<size_t>(t) * p.H + head) * p.D);
#pragma unroll
    for (int j = 0; j < CPL; ++j)
      if (lane + 32 * j < chunks) __stcs(dst + lane + 32 * j, pack8_bf16(f[j]));
    return;
  }
  const int64_t slot = static_cast<int64_t>(st) * p.win + pos % p.win;
  if (slot >= p.swa_pages) {
    if (lane == 0) atomicOr(p.status, 2);
    return;
  }
  if constexpr (FP8) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const int e = fp8_scale_exponent(amax);
    const float inv_scale = __int_as_float((127 - e) << 23);  // 2^-e, exact (e in [-126, 127])
    uint2* dst = reinterpret_cast<uint2*>(p.pool_fp8 + static_cast<size_t>(slot) * p.D);
#pragma unroll
    for (int j = 0; j < CPL; ++j) {
      if (lane + 32 * j < chunks) {
#pragma unroll
        for (int k = 0; k < 8; ++k) f[j][k] *= inv_scale;
        dst[lane + 32 * j] = pack8_e4m3(f[j]);
      }
    }
    if (lane == 0) p.pool_scale[slot] = __int_as_float((127 + e) << 23);
  } else {
    uint4* dst = reinterpret_cast<uint4*>(p.pool + static_cast<size_t>(slot) * p.D);
#pragma unroll
    for (int j = 0; j < CPL; ++j)
      if (lane + 32 * j < chunks) dst[lane + 32 * j] = pack8_bf16(f[j]);
  }
}

// A warp owns one row at a time and walks the rows grid-stride (measured
// best: one row per warp, 4-5 CTAs = 32-40 warps per SM; more rows per warp cost
// warps).  The state slot and position of the next row are requested one row
// ahead, so that a row's load and (LASTJ) its RoPE factor loads go out
// together: one memory latency per row rather than a position load followed
// by a dependent cache load.  The row -> (token, head) split is advanced
// incrementally (one division per thread).
template <int CPL>
constexpr int store_ctas_per_sm() { return CPL <= 2 ? 4 : 2; }  // 64 / 128 registers a thread

template <int CPL, bool FP8, bool LASTJ>
__global__ void __launch_bounds__(kStoreThreads, store_ctas_per_sm<CPL>())
    qk_norm_rope_store_kernel(StoreParams p) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int chunks = p.D >> 3;
  const int rope_chunk0 = (p.D - p.R) >> 3;
  const int half = p.R >> 1;
  const int rows = static_cast<int>(p.rows);
  const int rpt = p.H + 1;  // rows per token
  const int stride = static_cast<int>((gridDim.x * kStoreThreads) >> 5);
  const int stride_t = stride / rpt, stride_h = stride - stride_t * rpt;
  int row = static_cast<int>((blockIdx.x * kStoreThreads + threadIdx.x) >> 5);
  int t = row / rpt, head = row - t * rpt;
  int st = row < rows ? __ldg(p.state_slot + t) : -1;
  int pos = row < rows ? __ldg(p.positions + t) : -1;
  for (; row < rows; row += stride) {
    const uint16_t* src = head < p.H ? p.q + (static_cast<size_t>(t) * p.H + head) * p.D
                                     : p.kv + static_cast<size_t>(t) * p.D;
    uint4 x[CPL];
#pragma unroll
    for (int j = 0; j < CPL; ++j) {
      const int c = lane + 32 * j;
      x[j] = c < chunks ? __ldcs(reinterpret_cast<const uint4*>(src) + c) : make_uint4(0, 0, 0, 0);
    }
    float4 cs = make_float4(0.f, 0.f, 0.f, 0.f), sn = cs;
    if (LASTJ) {
      const int c = lane + 32 * (CPL - 1);
      if (st >= 0 && pos >= 0 && pos < p.max_pos && c >= rope_chunk0 && c < chunks) {
        const size_t off = static_cast<size_t>(pos) * half + 4 * (c - rope_chunk0);
        cs = __ldg(reinterpret_cast<const float4*>(p.cos_cache + off));
        sn = __ldg(reinterpret_cast<const float4*>(p.sin_cache + off));
      }
    }
    // the next row's token, and its state slot and position
    int nt = t + stride_t, nh = head + stride_h;
    if (nh >= rpt) nh -= rpt, ++nt;
    const bool more = row + stride < rows;
    const int nst = more ? __ldg(p.state_slot + nt) : -1;
    const int npos = more ? __ldg(p.positions + nt) : -1;
    process_row<CPL, FP8, LASTJ>(p, lane, x, t, head, st, pos, cs, sn);
    t = nt, head = nh, st = nst, pos = npos;
  }
  pdl_trigger();
}

template <int CPL, bool FP8, bool LASTJ>
cudaError_t launch_variant(const StoreParams& p, int num_sms, cudaStream_t st) {
  const int64_t want = (p.rows * 32 + kStoreThreads - 1) / kStoreThreads;  // a warp per row
  const int64_t cap = static_cast<int64_t>(num_sms) * store_ctas_per_sm<CPL>();
  const int grid = static_cast<int>(want < cap ? want : cap);
  return launch_pdl(qk_norm_rope_store_kernel<CPL, FP8, LASTJ>, dim3(grid),
                    dim3(kStoreThreads), 0, st, p);
}

template <int CPL, bool FP8>
cudaError_t launch_cpl(const StoreParams& p, int num_sms, cudaStream_t st) {
  const bool lastj = p.D % 256 == 0 && p.R <= 256;  // rotated dims all in chunk CPL-1
  return lastj ? launch_variant<CPL, FP8, true>(p, num_sms, st)
               : launch_variant<CPL, FP8, false>(p, num_sms, st);
}

}  // namespace

cudaError_t launch_qk_norm_rope_store(const void* q, const void* kv, const void* q_norm_w,
                                      const void* kv_norm_w, const float* cos_cache,
                                      const float* sin_cache, int max_pos,
                                      const int32_t* positions, const int32_t* state_slot, int N,
                                      int H, int D, int R, float eps, int win, int64_t swa_pages,
                                      void* q_out, void* pool, uint8_t* pool_fp8,
                                      float* pool_scale, int32_t* status, int num_sms,
                                      cudaStream_t st) {
  if (N == 0) return cudaSuccess;
  StoreParams p;
  p.q = static_cast<const uint16_t*>(q);
  p.kv = static_cast<const uint16_t*>(kv);
  p.q_norm_w = static_cast<const uint16_t*>(q_norm_w);
  p.kv_norm_w = static_cast<const uint16_t*>(kv_norm_w);
  p.cos_cache = cos_cache;
  p.sin_cache = sin_cache;
  p.positions = positions;
  p.state_slot = state_slot;
  p.q_out = static_cast<uint16_t*>(q_out);
  p.pool = static_cast<uint16_t*>(pool);
  p.pool_fp8 = pool_fp8;
  p.pool_scale = pool_scale;
  p.status = status;
  p.rows = static_cast<int64_t>(N) * (H + 1);
  p.swa_pages = swa_pages;
  p.N = N;
  p.H = H;
  p.D = D;
  p.R = R;
  p.max_pos = max_pos;
  p.win = win;
  p.eps = eps;
  const bool fp8 = pool_fp8 != nullptr;
  const int cpl = (D / 8 + 31) / 32;
#define SDA_STORE(C)                                                              \
  return fp8 ? launch_cpl<C, true>(p, num_sms, st) : launch_cpl<C, false>(p, num_sms, st)
  if (cpl <= 1) SDA_STORE(1);
  if (cpl <= 2) SDA_STORE(2);
  if (cpl <= 4) SDA_STORE(4);
  SDA_STORE(8);
#undef SDA_STORE
}

}  // namespace sda
