// sda_decode_simt.cu -- CUDA-core decode kernel for shapes the tensor-core
// kernel does not take (D < 512, or H not a multiple of 16 / 64).
//
// One warp per head; the lanes split D, each slot row is read with 16-byte
// (or narrower) vector loads, the dot products are finished with butterfly
// shuffles and the softmax runs online in the log2 domain in fp32, with the
// sink merged into the denominator at the end (paged_decode.py docstring,
// "numerics").  Slots are processed four at a time to overlap the loads and
// the shuffle reductions.
#include <cuda_bf16.h>

#include "sda_internal.cuh"

namespace sda {

namespace {

constexpr int kSimtThreads = 256;
constexpr int kSimtWarps = kSimtThreads / 32;
constexpr int kSlotsPerStep = 4;

template <int D>
struct LaneShape {
  static constexpr int kVec = D / 32 >= 8 ? 8 : D / 32;  // bf16 per vector load
  static constexpr int kNv = D / (32 * kVec);            // vectors per lane
  static constexpr int kPer = kVec * kNv;                // elements per lane
};

template <int VEC>
__device__ __forceinline__ void load_bf16(const __nv_bfloat16* p, float* v) {
  if constexpr (VEC == 8) {
    uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 f = __bfloat1622float2(h[i]);
      v[2 * i] = f.x;
      v[2 * i + 1] = f.y;
    }
  } else if constexpr (VEC == 4) {
    uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      float2 f = __bfloat1622float2(h[i]);
      v[2 * i] = f.x;
      v[2 * i + 1] = f.y;
    }
  } else {
    static_assert(VEC == 2, "vector width");
    uint32_t u = __ldg(reinterpret_cast<const unsigned int*>(p));
    float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u));
    v[0] = f.x;
    v[1] = f.y;
  }
}

template <int VEC>
__device__ __forceinline__ void store_bf16(__nv_bfloat16* p, const float* v) {
  if constexpr (VEC == 8) {
    uint4 u;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    *reinterpret_cast<uint4*>(p) = u;
  } else if constexpr (VEC == 4) {
    uint2 u;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 2; ++i) h[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    *reinterpret_cast<uint2*>(p) = u;
  } else {
    __nv_bfloat162 h = __floats2bfloat162_rn(v[0], v[1]);
    *reinterpret_cast<__nv_bfloat162*>(p) = h;
  }
}

template <int D>
__global__ void __launch_bounds__(kSimtThreads)
decode_simt_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ kv,
                   const int32_t* __restrict__ kv_indices, const float* __restrict__ attn_sink,
                   float qk_scale_log2, int H, __nv_bfloat16* __restrict__ out,
                   const int* __restrict__ cta_start, const int4* __restrict__ units,
                   float2* __restrict__ part_ml, float* __restrict__ part_o) {
  using S = LaneShape<D>;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  pdl_wait();
  pdl_trigger();
  // this CTA's run of the unit list
  const int u0 = cta_start[blockIdx.x], u1 = cta_start[blockIdx.x + 1];
  for (int pos = u0; pos < u1; ++pos) {
    const int4 u = units[pos];
    const int t = u.x, begin = u.y, len = u.z, row = unit_part_row(u.w);
    for (int h = warp; h < H; h += kSimtWarps) {
      const size_t qo = ((size_t)t * H + h) * D;
      float qv[S::kPer], acc[S::kPer];
#pragma unroll
      for (int v = 0; v < S::kNv; ++v)
        load_bf16<S::kVec>(q + qo + v * 32 * S::kVec + lane * S::kVec, qv + v * S::kVec);
#pragma unroll
      for (int e = 0; e < S::kPer; ++e) acc[e] = 0.f;
      float m = -INFINITY, l = 0.f;
      for (int j0 = 0; j0 < len; j0 += kSlotsPerStep) {
        const int nj = min(kSlotsPerStep, len - j0);
        float kvv[kSlotsPerStep][S::kPer];
        float s[kSlotsPerStep];
#pragma unroll
        for (int j = 0; j < kSlotsPerStep; ++j) {
          const int jj = j < nj ? j : 0;  // tail: reload a valid row, weight forced to 0 below
          const __nv_bfloat16* r = kv + (size_t)kv_indices[begin + j0 + jj] * D;
#pragma unroll
          for (int v = 0; v < S::kNv; ++v)
            load_bf16<S::kVec>(r + v * 32 * S::kVec + lane * S::kVec, kvv[j] + v * S::kVec);
          float d = 0.f;
#pragma unroll
          for (int e = 0; e < S::kPer; ++e) d = fmaf(qv[e], kvv[j][e], d);
          s[j] = d;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
#pragma unroll
          for (int j = 0; j < kSlotsPerStep; ++j) s[j] += __shfl_xor_sync(0xffffffffu, s[j], o);
        float mx = m;
#pragma unroll
        for (int j = 0; j < kSlotsPerStep; ++j) {
          s[j] = j < nj ? s[j] * qk_scale_log2 : -INFINITY;
          mx = fmaxf(mx, s[j]);
        }
        const float alpha = ex2_approx(m - mx);  // m = -inf on the first step -> 0
        l *= alpha;
#pragma unroll
        for (int e = 0; e < S::kPer; ++e) acc[e] *= alpha;
#pragma unroll
        for (int j = 0; j < kSlotsPerStep; ++j) {
          const float p = ex2_approx(s[j] - mx);
          l += p;
#pragma unroll
          for (int e = 0; e < S::kPer; ++e) acc[e] = fmaf(p, kvv[j][e], acc[e]);
        }
        m = mx;
      }
      if (row < 0) {
        // finish the token: merge the sink (virtual key, zero value)
        const float ms = attn_sink[h] * kLog2e;
        const float M = fmaxf(m, ms);
        float f = 0.f;
        if (M != -INFINITY && ms != INFINITY) {
          const float a = ex2_approx(m - M);
          const float den = l * a + ex2_approx(ms - M);
          f = a / den;
        }
        float o[S::kPer];
#pragma unroll
        for (int e = 0; e < S::kPer; ++e) o[e] = acc[e] * f + 0.f;  // -0 -> +0 when f = 0
#pragma unroll
        for (int v = 0; v < S::kNv; ++v)
          store_bf16<S::kVec>(out + qo + v * 32 * S::kVec + lane * S::kVec, o + v * S::kVec);
      } else {
        float* po = part_o + ((size_t)row * H + h) * D;
#pragma unroll
        for (int v = 0; v < S::kNv; ++v)
#pragma unroll
          for (int e = 0; e < S::kVec; ++e) po[v * 32 * S::kVec + lane * S::kVec + e] = acc[v * S::kVec + e];
        if (lane == 0) part_ml[(size_t)row * H + h] = make_float2(m, l);
      }
    }
  }
}

template <int D>
cudaError_t launch_simt_d(const void* q, const void* kv, const int32_t* kv_indices,
                          const float* attn_sink, float scale, int H, void* out, void* ws,
                          const WsLayout& L, const LaunchPlan& lp, cudaStream_t st) {
  char* base = static_cast<char*>(ws);
  return launch_pdl(decode_simt_kernel<D>, dim3(lp.grid), dim3(kSimtThreads), 0, st,
                    static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(kv),
                    kv_indices, attn_sink, scale * kLog2e, H, static_cast<__nv_bfloat16*>(out),
                    reinterpret_cast<const int*>(base + L.cta_off),
                    reinterpret_cast<const int4*>(base + L.units_off),
                    reinterpret_cast<float2*>(base + L.ml_off),
                    reinterpret_cast<float*>(base + L.o_off));
}

}  // namespace

cudaError_t launch_decode_simt(const void* q, const void* kv, const int32_t* kv_indices,
                               const float* attn_sink, float softmax_scale, int N, int H, int D,
                               void* out, void* ws, const WsLayout& L, const LaunchPlan& lp,
                               cudaStream_t st) {
  (void)N;
  switch (D) {
    case 64: return launch_simt_d<64>(q, kv, kv_indices, attn_sink, softmax_scale, H, out, ws, L, lp, st);
    case 128: return launch_simt_d<128>(q, kv, kv_indices, attn_sink, softmax_scale, H, out, ws, L, lp, st);
    case 256: return launch_simt_d<256>(q, kv, kv_indices, attn_sink, softmax_scale, H, out, ws, L, lp, st);
    case 512: return launch_simt_d<512>(q, kv, kv_indices, attn_sink, softmax_scale, H, out, ws, L, lp, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace sda
