// sda_decode_pair.cu -- two-CTA (thread-block cluster) tensor-core decode
// kernel for D = 512 and NH = 16, 32 or 64 heads per unit (H = 128 runs as
// two head groups).
//
// What it computes is the paged_decode.py docstring quoted on the sglang
// PR 28392 summary page ("关键源码片段": caller convention, returns,
// numerics): for each token t and head h, attention of q[t,h] over the rows
// unified_kv[kv_indices[kv_indptr[t]:kv_indptr[t+1]]] -- each row is both key
// and value -- with the per-head sink as a virtual key of zero value, an
// fp32 online softmax in the log2 domain, out in bf16.
//
// Design for GB300 (not from the page, whose kernel targets AMD GPUs).
// Every tcgen05.mma of the shapes a decode step allows costs about the same
// time on this GPU (~72 cycles measured for M = 64 or 128 and N <= 128), so
// the kernel is built to issue few, wide MMAs:
//  * A cluster of two CTAs (on two SMs) owns one work unit at a time.  CTA r
//    holds columns [256r, 256r + 256) of D: of q, of every KV row it
//    gathers, and of the output.  A tile is 128 slots, i.e. 64 KB of
//    half-rows per CTA, in 2 shared-memory stages.
//  * S = Q K^T over the CTA's half of D: M = 64 (padded heads), N = 128
//    slots, K = 256 -- 16 MMAs per tile.  The two partial score tiles are
//    exchanged through distributed shared memory, so that both CTAs hold
//    the full S and run identical softmaxes (same maxima, same rounding):
//    each CTA then needs only its own half of V.
//  * O^T += V^T P^T over the CTA's half of D: M = 128 rows of D, N = NH
//    heads, K = 16 slots -- 16 MMAs per tile.
//  * Warps 8..15 gather half-rows (one 512-byte load per warp and row, 16
//    rows of a tile per warp in flight), warp 16 issues the QK MMAs and the
//    q loads (tiled TMA), warp 17 the PV MMAs (18 and 19 only fill out the
//    register split, see kThreads); warps 0..7 run the softmax:
//    warps q and q + 4 share TMEM lane quadrant q and take slots 0..63 and
//    64..127 of each tile, combining their halves' maxima through shared
//    memory.  The lazy rescale of the running max (only when it grows by
//    more than 8 in log2 units, so p <= 256) is decided from the full S and
//    therefore identically in both CTAs.
//  * Every mbarrier wait is bounded (2 s); on timeout the kernel raises the
//    workspace error word, drains its own copies and returns.  A CTA never
//    leaves before its partner (cluster barrier at the end), so remote
//    stores and arrivals always find live shared memory.
#include <cuda.h>
#include <cuda_bf16.h>

#include "sda_internal.cuh"
#include "umma_ptx.cuh"

namespace sda {

namespace {

using namespace ptx;

constexpr int kD = 512;
constexpr int kHalf = kD / 2;               // columns of D per CTA
constexpr int kTile = kPairTileSlots;       // 128 slots per tile
constexpr int kPanels = kHalf / 64;         // 4 column panels of 128 bytes per half-row
constexpr int kPanelKV = kTile * 128;       // 16 KB
constexpr int kKVBytes = kPanels * kPanelKV;  // 64 KB per stage
constexpr int kSmWarps = 8;                 // warps 0..7: softmax / epilogue
constexpr int kSmThreads = kSmWarps * 32;
constexpr int kLoaderWarp0 = 8;             // warps 8..15: KV half-row loaders
constexpr int kLoaderWarps = 8;
constexpr int kRowsPerLoader = kTile / kLoaderWarps;  // 16
constexpr int kQkWarp = 16;                 // QK issuer + q loads
constexpr int kPvWarp = 17;                 // PV issuer
// 20 warps (18, 19 idle): warps are spread over the SM's four sub-partitions
// and each sub-partition has 16 K registers, so 18 or 20 warps (5 on some
// sub-partitions) leave at most 96 registers per thread.
constexpr int kThreads = 20 * 32;
constexpr int kMaxRegs = 96;
constexpr float kRescaleThreshold = 8.0f;   // log2 units
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;
static_assert(kRowsPerLoader <= 32, "slot indices of a warp's rows live in one register per lane");

enum Bar : int {
  kBarQFull = 0,
  kBarQEmpty,
  kBarOEmpty,
  kBarDrain,
  kBarDrainPv,
  kBarRecvFull,   // the partner's partial S of this tile has landed here
  kBarRecvFree,   // the partner has consumed the partial S this CTA sent it
  kBarKVFull0,    // 2 stages
  kBarPVDone0 = kBarKVFull0 + 2,
  kBarSFull0 = kBarPVDone0 + 2,   // 2 S buffers
  kBarSEmpty0 = kBarSFull0 + 2,
  kBarPFull0 = kBarSEmpty0 + 2,   // 2 P buffers
  kNumBars = kBarPFull0 + 2
};

// named barriers (id 0 is __syncthreads)
constexpr int kNbSoftmax = 1;     // all 256 softmax threads
constexpr int kNbPair0 = 2;       // 2..5: warps q and q + 4 (64 threads)
constexpr int kNbBlock0 = 6;      // 6..7: the 4 warps writing O^T block b (128 threads)

template <int NH>
struct PCfg {
  static constexpr int kNW = NH / 16;            // TMEM quadrants holding real heads
  static constexpr int kXWarps = 2 * kNW;        // softmax warps that exchange partial S
  static constexpr int kPanelQ = NH * 128;       // q rows are packed NH apart (see below)
  static constexpr int kQBytes = kPanels * kPanelQ;
  static constexpr int kPBytes = 2 * NH * 128;   // P: 2 atoms of 64 slots x NH rows x 128 B
  static constexpr int kRecvBytes = kXWarps * 8 * 32 * 16;  // 32 floats per exchanging thread
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = kQBytes;
  static constexpr int kOffP = kOffKV + 2 * kKVBytes;
  static constexpr int kOffRecv = kOffP + 2 * kPBytes;
  static constexpr int kOffBar = kOffRecv + kRecvBytes;
  static constexpr int kOffMisc = kOffBar + 192;
  // misc: tmem base (4), abort flag (4), pad; then per-head float arrays.
  // alpha (rescale factors, used inside a unit's tiles) and fac (output
  // factors, used in its epilogue) share one array: named barriers separate
  // every use of one from every use of the other.
  static constexpr int kOffAlpha = kOffMisc + 16;       // [64]
  static constexpr int kOffFac = kOffAlpha;             // [64]
  static constexpr int kOffHMax = kOffAlpha + 4 * 64;   // [2 tiles][2 halves][64]
  static constexpr int kOffLSum = kOffHMax + 4 * 256;   // [2 halves][64]
  static constexpr int kSmemUsed = kOffLSum + 4 * 128;
  static constexpr int kSmem = kSmemUsed + 1024;        // slack for 1024-byte alignment
  static constexpr int kOCol = 256;  // S buffers at columns 0 and 128; O^T block b at [256 + b*NH, +NH)
  static constexpr int kTmemCols = 512;
  static constexpr uint32_t kIdescQK = idesc_bf16_f32(64, kTile, false, false);
  static constexpr uint32_t kIdescPV = idesc_bf16_f32(128, NH, true, false);
  static_assert(kOffKV % 1024 == 0 && kPanelQ % 1024 == 0 && kOffP % 1024 == 0, "1 KB atoms");
  // the QK MMA reads 64 rows per q panel; rows NH..63 are whatever follows
  // (other panels, then the first KV stage): valid shared memory whose
  // products land in TMEM lanes that nothing reads
  static_assert((kPanels - 1) * kPanelQ + 64 * 128 <= kOffBar, "padded A operand inside smem");
  static_assert(kNumBars * 8 <= 192, "mbarrier area");
  static_assert(kSmem <= 232448, "shared memory budget");
  static_assert(kOCol + 2 * NH <= kTmemCols, "TMEM columns");
  static_assert(2 * kPBytes >= 2 * NH * 256, "P buffers hold the two output staging blocks");
};

struct Params {
  const __nv_bfloat16* kv;
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

// Bounded wait (see the one-CTA kernel): false on timeout or once this CTA
// has aborted.  `cluster` selects a cluster-scope acquire, needed where the
// phase was completed by the partner CTA's arrivals.
template <bool cluster = false>
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         WsHeader* hdr) {
  auto probe = [&]() { return cluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity); };
  if (probe()) return true;
  if (*abort_flag) return false;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (probe()) return true;
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

__device__ __forceinline__ void drain_bar(uint32_t bar, uint32_t parity, WsHeader* hdr) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kWaitTimeoutNs) {
      atomicExch(&hdr->error, 1);
      return;
    }
  }
}

// Walks the tiles of the units a cluster owns, in the same order in every
// role of both CTAs: unit k of pair c is unit_position(k, c, pairs).
struct TileCursor {
  const int4* units;
  int n_units, pair, pairs;
  int k;       // unit slot in the pair's sequence
  int4 u;      // current unit
  int ntiles;  // tiles of the current unit
  int i;       // tile within the unit
  int g;       // tiles seen before this one (all units)
  int nu;      // units with slots seen before this one
  bool valid;
  __device__ __forceinline__ int len() const { return u.z; }
  __device__ __forceinline__ void seek() {
    for (;; ++k) {
      const int pos = unit_position(k, pair, pairs);
      if (pos >= n_units) {
        valid = false;
        return;
      }
      u = units[pos];
      if (u.z > 0) {
        ntiles = (u.z + kTile - 1) / kTile;
        i = 0;
        valid = true;
        return;
      }
    }
  }
  __device__ __forceinline__ void init(const int4* us, int n) {
    units = us;
    n_units = n;
    pair = blockIdx.x >> 1;
    pairs = gridDim.x >> 1;
    k = 0;
    g = 0;
    nu = 0;
    seek();
  }
  __device__ __forceinline__ void next() {
    ++g;
    if (++i == ntiles) {
      ++nu;
      ++k;
      seek();
    }
  }
};

template <int NH>
__global__ void __cluster_dims__(2, 1, 1) __maxnreg__(kMaxRegs)
decode_pair_kernel(const __grid_constant__ CUtensorMap tmap_q,
                   const __grid_constant__ CUtensorMap tmap_out, const Params p) {
  using C = PCfg<NH>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_addr(smem);
  const uint32_t sQ = sbase + C::kOffQ;
  const uint32_t sKV = sbase + C::kOffKV;
  const uint32_t sP = sbase + C::kOffP;
  const uint32_t sRecv = sbase + C::kOffRecv;
  const uint32_t sBar = sbase + C::kOffBar;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
  float* s_alpha = reinterpret_cast<float*>(smem + C::kOffAlpha);
  float* s_fac = reinterpret_cast<float*>(smem + C::kOffFac);
  float* s_hmax = reinterpret_cast<float*>(smem + C::kOffHMax);
  float* s_lsum = reinterpret_cast<float*>(smem + C::kOffLSum);
  auto bar = [&](int i) { return sBar + 8u * (uint32_t)i; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;

  if (threadIdx.x == 0) {
    mbar_init(bar(kBarQFull), 1);
    mbar_init(bar(kBarQEmpty), 1);
    mbar_init(bar(kBarOEmpty), kSmWarps);
    mbar_init(bar(kBarDrain), 1);
    mbar_init(bar(kBarDrainPv), 1);
    mbar_init(bar(kBarRecvFull), C::kXWarps);
    mbar_init(bar(kBarRecvFree), C::kXWarps);
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(kBarKVFull0 + b), kLoaderWarps);
      mbar_init(bar(kBarPVDone0 + b), 1);
      mbar_init(bar(kBarSFull0 + b), 1);
      mbar_init(bar(kBarSEmpty0 + b), kSmWarps);
      mbar_init(bar(kBarPFull0 + b), kSmWarps);
    }
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmap_q);
    tma_prefetch_desc(&tmap_out);
  }
  if (warp == kQkWarp) {
    tmem_alloc(smem_addr(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync_all();  // the partner's barriers are initialised before any remote arrival
  const uint32_t tmem = *tmem_slot;
  // everything above overlaps the previous kernel (PDL); global memory only below
  pdl_wait();
  pdl_trigger();
  const int n_units = p.hdr->n_units;
  const int H = p.H;

  if (warp >= kLoaderWarp0 && warp < kLoaderWarp0 + kLoaderWarps) {
    // ===================================================== KV half-row loaders
    // Loader warp w owns rows [16w, 16w+16) of every tile; each row's 512
    // bytes (this CTA's half of D) are one 16-byte load per lane, so a
    // thread keeps 16 loads and an SM 64 KB in flight.  A tile's loads are
    // issued before the warp waits for its stage; kv_indices one tile ahead.
    const int lw = warp - kLoaderWarp0;
    const uint4* kv4 = reinterpret_cast<const uint4*>(p.kv) + rank * (kHalf / 8);
    TileCursor cur;
    cur.init(p.units, n_units);
    auto fetch_slots = [&]() -> int {  // lanes 0..15: slot of row 16w + lane (-1: none)
      if (!cur.valid) return -1;
      const int n = min(kTile, cur.len() - cur.i * kTile);
      const int r = lw * kRowsPerLoader + lane;
      return (lane < kRowsPerLoader && r < n) ? __ldg(p.kv_indices + cur.u.y + cur.i * kTile + r) : -1;
    };
    uint4 v[kRowsPerLoader];
    auto issue = [&](int slots) {
#pragma unroll
      for (int r = 0; r < kRowsPerLoader; ++r) {
        const int slot = __shfl_sync(0xffffffffu, slots, r);
        v[r] = slot >= 0 ? __ldcg(kv4 + (size_t)slot * (kD / 8) + lane) : make_uint4(0, 0, 0, 0);
      }
    };
    auto store = [&](int g) -> bool {
      const int s = g & 1;
      if (g >= 2) {  // the stage is free once the PV of tile g - 2 is done
        bool ok = true;
        if (lane == 0) ok = wait_bar(bar(kBarPVDone0 + s), ((g >> 1) - 1) & 1, abort_flag, p.hdr);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) return false;
      }
      uint8_t* stage = smem + C::kOffKV + s * kKVBytes;
      const int c = lane >> 3, k = lane & 7;  // 16-byte chunk `lane` of the half-row: panel c, chunk k
#pragma unroll
      for (int r = 0; r < kRowsPerLoader; ++r) {
        const int row = lw * kRowsPerLoader + r;
        *reinterpret_cast<uint4*>(stage + c * kPanelKV + (row >> 3) * 1024 + (row & 7) * 128 +
                                  ((k ^ (row & 7)) << 4)) = v[r];
      }
      fence_proxy_async_smem();  // generic-proxy stores -> read by the tensor cores
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarKVFull0 + s));
      return true;
    };
    if (cur.valid) {
      int g = cur.g;
      issue(fetch_slots());
      cur.next();
      int next_slots = fetch_slots();
      while (store(g) && cur.valid) {
        g = cur.g;
        issue(next_slots);
        cur.next();
        next_slots = fetch_slots();
      }
    }
  } else if (warp == kQkWarp || warp == kPvWarp) {
    // ===================================================== MMA issuers
    //  - warp 16, lane 0: partial S = Q K^T of every tile as soon as the
    //    tile has landed and its S buffer is free; q of the next unit (tiled
    //    TMA, this CTA's half of D) once this unit's last QK has read q;
    //  - warp 17, lane 0: O^T += V^T P^T as soon as P is written (its commit
    //    frees the KV stage and the P buffer).
    if (lane == 0) {
      const bool qk_role = warp == kQkWarp;
      TileCursor cq;
      cq.init(p.units, n_units);
      int q_issued = 0;
      bool ok = true;
      auto load_q = [&]() {
        mbar_arrive_expect_tx(bar(kBarQFull), NH * 128 * kPanels);
        const int qrow = cq.u.x * H + unit_head_group(cq.u.w) * NH;
#pragma unroll
        for (int c = 0; c < kPanels; ++c)
          tma_load_2d(sQ + c * C::kPanelQ, &tmap_q, (int)rank * kHalf + c * 64, qrow, bar(kBarQFull));
      };
      if (qk_role && cq.valid) {
        load_q();
        q_issued = 1;
      }
      while (cq.valid && ok) {
        const int g = cq.g, s = g & 1;
        const uint32_t kvs = sKV + s * kKVBytes;
        if (qk_role) {
          ok = wait_bar(bar(kBarKVFull0 + s), (g >> 1) & 1, abort_flag, p.hdr);
          if (ok && g >= 2) ok = wait_bar(bar(kBarSEmpty0 + s), ((g >> 1) - 1) & 1, abort_flag, p.hdr);
          if (ok && cq.i == 0) ok = wait_bar(bar(kBarQFull), cq.nu & 1, abort_flag, p.hdr);
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < kPanels; ++c) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t a = sdesc_sw128(sQ + c * C::kPanelQ + kk * 32, 16, 1024);
              const uint64_t bd = sdesc_sw128(kvs + c * kPanelKV + kk * 32, 16, 1024);
              mma_bf16(tmem + s * kTile, a, bd, C::kIdescQK, (c | kk) ? 1u : 0u);
            }
          }
          mma_commit(bar(kBarSFull0 + s));
          const bool last = cq.i == cq.ntiles - 1;
          const int nu = cq.nu;
          if (last) mma_commit(bar(kBarQEmpty));
          cq.next();
          if (last && cq.valid) {
            ok = wait_bar(bar(kBarQEmpty), nu & 1, abort_flag, p.hdr);
            if (!ok) break;
            load_q();
            q_issued = cq.nu + 1;
          }
        } else {
          const bool first = cq.i == 0;
          ok = wait_bar(bar(kBarPFull0 + s), (g >> 1) & 1, abort_flag, p.hdr);
          if (ok && first && cq.nu >= 1) ok = wait_bar(bar(kBarOEmpty), (cq.nu - 1) & 1, abort_flag, p.hdr);
          if (!ok) break;
          tc_fence_after();
          const uint32_t ps = sP + s * C::kPBytes;
#pragma unroll
          for (int b = 0; b < 2; ++b) {
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk) {
              // A = V^T block b: rows d of panels 2b, 2b+1 (MN-major), K = slots [16kk, 16kk+16)
              const uint64_t a = sdesc_sw128(kvs + (2 * b) * kPanelKV + kk * 2048, kPanelKV, 1024);
              // B = P^T: N = NH head rows, K = 16 slots of atom kk/4 at byte 32*(kk%4)
              const uint64_t bd = sdesc_sw128(ps + (kk >> 2) * (NH * 128) + (kk & 3) * 32, 16, 1024);
              mma_bf16(tmem + C::kOCol + b * NH, a, bd, C::kIdescPV, (first && kk == 0) ? 0u : 1u);
            }
          }
          mma_commit(bar(kBarPVDone0 + s));
          cq.next();
        }
      }
      const int drain = qk_role ? kBarDrain : kBarDrainPv;
      mma_commit(bar(drain));
      drain_bar(bar(drain), 0, p.hdr);
      if (qk_role && q_issued >= 1) drain_bar(bar(kBarQFull), (q_issued - 1) & 1, p.hdr);
    }
    __syncwarp();
  } else if (warp < kSmWarps) {
    // ===================================================== softmax + epilogue
    // Warp w reads TMEM lane quadrant q = w % 4 and slots [64*hc, 64*hc + 64)
    // of each tile, hc = w / 4, with the 16x256b shape: thread t holds heads
    // hA = 16q + t/4 and hB = hA + 8 (the M = 64 accumulator keeps row r in
    // lane 32*(r/16) + r%16) for the 16 slots 64hc + 8rep + 2(t%4) + {0,1}.
    const int q4 = warp & 3, hc = warp >> 2;
    const int st = threadIdx.x;  // 0..255
    const int tq = lane & 3;
    const int hA = q4 * 16 + (lane >> 2), hB = hA + 8;
    const bool vA = hA < NH, vB = hB < NH;
    const bool xw = q4 < C::kNW;  // this warp's heads are real: it exchanges partial S
    const int xi = hc * C::kNW + q4;  // its slot in the exchange buffers
    const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
    const float sc = p.qk_scale_log2;
    const bool pos_sc = sc >= 0.f;
    const uint32_t recv_mine = sRecv + (uint32_t)(((xi * 8) * 32 + lane) * 16);
    const uint32_t recv_peer = mapa_shared(recv_mine, peer);
    const uint32_t peer_recv_full = mapa_shared(bar(kBarRecvFull), peer);
    const uint32_t peer_recv_free = mapa_shared(bar(kBarRecvFree), peer);
    // Control flow is identical in the eight warps (it depends only on the
    // unit list and on block-wide votes), so every named barrier is reached
    // by all of them even after a wait timed out.
    int g = 0;
    const int pair = blockIdx.x >> 1, pairs = gridDim.x >> 1;
    for (int k = 0;; ++k) {
      const int pos = unit_position(k, pair, pairs);
      if (pos >= n_units) break;
      const int4 u = p.units[pos];
      const int t = u.x, len = u.z, hg = unit_head_group(u.w), row = unit_part_row(u.w);
      if (len <= 0) {
        // padded token: out = 0 for this CTA's half of D of its NH heads
        for (int e = st; e < NH * (kHalf / 8); e += kSmThreads) {
          const int h = e / (kHalf / 8), c = e % (kHalf / 8);
          reinterpret_cast<uint4*>(p.out + ((size_t)t * H + hg * NH + h) * kD + rank * kHalf)[c] =
              make_uint4(0, 0, 0, 0);
        }
        continue;
      }
      const int ntiles = (len + kTile - 1) / kTile;
      float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;  // l: this thread's share
      for (int i = 0; i < ntiles; ++i, ++g) {
        const int s = g & 1;
        const int n = min(kTile, len - i * kTile);
        wait_bar(bar(kBarSFull0 + s), (g >> 1) & 1, abort_flag, p.hdr);
        tc_fence_after();
        uint32_t sv[32];
        tmem_ld_16x256b_x8(tmem + lane_base + s * kTile + 64 * hc, sv);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarSEmpty0 + s));  // S buffer s may be overwritten
        if (xw) {
          // send this partial to the partner (once it has consumed the last
          // one), then add the partner's partial of the same elements
          if (g >= 1) {
            if (lane == 0) wait_bar<true>(bar(kBarRecvFree), (g - 1) & 1, abort_flag, p.hdr);
            __syncwarp();
          }
#pragma unroll
          for (int c = 0; c < 8; ++c)
            st_cluster_v4(recv_peer + c * 512, sv[4 * c], sv[4 * c + 1], sv[4 * c + 2], sv[4 * c + 3]);
          __syncwarp();
          if (lane == 0) mbar_arrive_remote(peer_recv_full);
          if (lane == 0) wait_bar<true>(bar(kBarRecvFull), g & 1, abort_flag, p.hdr);
          __syncwarp();
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const float4 o = *reinterpret_cast<const float4*>(smem + (recv_mine - sbase) + c * 512);
            sv[4 * c + 0] = __float_as_uint(__uint_as_float(sv[4 * c + 0]) + o.x);
            sv[4 * c + 1] = __float_as_uint(__uint_as_float(sv[4 * c + 1]) + o.y);
            sv[4 * c + 2] = __float_as_uint(__uint_as_float(sv[4 * c + 2]) + o.z);
            sv[4 * c + 3] = __float_as_uint(__uint_as_float(sv[4 * c + 3]) + o.w);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive_remote(peer_recv_free);
        }
        // largest scaled logit per head over this warp's valid slots
        float eA = pos_sc ? -INFINITY : INFINITY, eB = eA;
#pragma unroll
        for (int rep = 0; rep < 8; ++rep) {
#pragma unroll
          for (int kk = 0; kk < 2; ++kk) {
            if (64 * hc + 8 * rep + 2 * tq + kk < n) {
              const float a = __uint_as_float(sv[4 * rep + kk]), b = __uint_as_float(sv[4 * rep + 2 + kk]);
              eA = pos_sc ? fmaxf(eA, a) : fminf(eA, a);
              eB = pos_sc ? fmaxf(eB, b) : fminf(eB, b);
            }
          }
        }
#pragma unroll
        for (int o = 1; o <= 2; o <<= 1) {
          const float xa = __shfl_xor_sync(0xffffffffu, eA, o), xb = __shfl_xor_sync(0xffffffffu, eB, o);
          eA = pos_sc ? fmaxf(eA, xa) : fminf(eA, xa);
          eB = pos_sc ? fmaxf(eB, xb) : fminf(eB, xb);
        }
        // combine with the other half of the tile (warp w ^ 4)
        {
          float* hm = s_hmax + (g & 1) * 128;
          if (tq == 0) {
            hm[hc * 64 + hA] = eA;
            hm[hc * 64 + hB] = eB;
          }
          named_bar_sync(kNbPair0 + q4, 64);
          const float oA = hm[(hc ^ 1) * 64 + hA], oB = hm[(hc ^ 1) * 64 + hB];
          eA = pos_sc ? fmaxf(eA, oA) : fminf(eA, oA);
          eB = pos_sc ? fmaxf(eB, oB) : fminf(eB, oB);
        }
        const float tA = eA * sc, tB = eB * sc;
        float alphaA = 1.f, alphaB = 1.f;
        bool need = false;
        if (vA && tA > mA + kRescaleThreshold) {
          alphaA = ex2_approx(mA - tA);  // 0 on the first tile (m = -inf)
          need = i > 0;
          lA *= alphaA;
          mA = tA;
        }
        if (vB && tB > mB + kRescaleThreshold) {
          alphaB = ex2_approx(mB - tB);
          need = need || i > 0;
          lB *= alphaB;
          mB = tB;
        }
        // P buffer s is free once the PV of tile g-2 is done
        if (g >= 2) {
          if (lane == 0) wait_bar(bar(kBarPVDone0 + s), ((g >> 1) - 1) & 1, abort_flag, p.hdr);
          __syncwarp();
        }
        // p = 2^(s*scale - m) in bf16 into rows hA, hB of P atom hc (K-major,
        // 128-byte swizzle: chunk `rep` of 8 slots at (rep ^ (h & 7)) * 16,
        // this thread's slot pair at byte 4*tq of the chunk)
        uint8_t* pbase = smem + C::kOffP + s * C::kPBytes + hc * (NH * 128);
        uint8_t* prowA = pbase + (hA >> 3) * 1024 + (hA & 7) * 128 + 4 * tq;
        uint8_t* prowB = pbase + (hB >> 3) * 1024 + (hB & 7) * 128 + 4 * tq;
        float sA = 0.f, sB = 0.f;
#pragma unroll
        for (int rep = 0; rep < 8; ++rep) {
          const int j = 64 * hc + 8 * rep + 2 * tq;
          const float a0 = j < n ? ex2_approx(fmaf(__uint_as_float(sv[4 * rep + 0]), sc, -mA)) : 0.f;
          const float a1 = j + 1 < n ? ex2_approx(fmaf(__uint_as_float(sv[4 * rep + 1]), sc, -mA)) : 0.f;
          const float b0 = j < n ? ex2_approx(fmaf(__uint_as_float(sv[4 * rep + 2]), sc, -mB)) : 0.f;
          const float b1 = j + 1 < n ? ex2_approx(fmaf(__uint_as_float(sv[4 * rep + 3]), sc, -mB)) : 0.f;
          __nv_bfloat162 pa = __floats2bfloat162_rn(a0, a1), pb = __floats2bfloat162_rn(b0, b1);
          // the denominator sums the same bf16 weights the PV MMA multiplies
          const float2 fa = __bfloat1622float2(pa), fb = __bfloat1622float2(pb);
          sA += fa.x + fa.y;
          sB += fb.x + fb.y;
          if (vA) *reinterpret_cast<uint32_t*>(prowA + ((rep ^ (hA & 7)) << 4)) = *reinterpret_cast<uint32_t*>(&pa);
          if (vB) *reinterpret_cast<uint32_t*>(prowB + ((rep ^ (hB & 7)) << 4)) = *reinterpret_cast<uint32_t*>(&pb);
        }
        lA += sA;
        lB += sB;
        fence_proxy_async_smem();
        if (named_bar_or(kNbSoftmax, kSmThreads, need)) {
          // some running max grew: scale O^T (this CTA's half of D) by alpha
          if (hc == 0 && tq == 0) {
            if (vA) s_alpha[hA] = alphaA;
            if (vB) s_alpha[hB] = alphaB;
          }
          named_bar_sync(kNbSoftmax, kSmThreads);
          // O^T must be quiescent: wait for the PV of tile g-1
          if (lane == 0) wait_bar(bar(kBarPVDone0 + ((g - 1) & 1)), ((g - 1) >> 1) & 1, abort_flag, p.hdr);
          __syncwarp();
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < NH / 16; ++c) {
            uint32_t ov[16];
            const uint32_t ta = tmem + lane_base + C::kOCol + hc * NH + c * 16;
            tmem_ld16(ta, ov);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * s_alpha[c * 16 + e]);
            tmem_st16(ta, ov);
          }
          tmem_wait_st();
          named_bar_sync(kNbSoftmax, kSmThreads);  // s_alpha is rewritten next time
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarPFull0 + s));
      }
      // ---------------------------------------------- epilogue of the unit
      // denominators: the quad's shares, then the two halves of the tile
      lA += __shfl_xor_sync(0xffffffffu, lA, 1);
      lA += __shfl_xor_sync(0xffffffffu, lA, 2);
      lB += __shfl_xor_sync(0xffffffffu, lB, 1);
      lB += __shfl_xor_sync(0xffffffffu, lB, 2);
      if (tq == 0) {
        s_lsum[hc * 64 + hA] = lA;
        s_lsum[hc * 64 + hB] = lB;
      }
      const int gl = g - 1;
      if (lane == 0) wait_bar(bar(kBarPVDone0 + (gl & 1)), (gl >> 1) & 1, abort_flag, p.hdr);
      __syncwarp();
      tc_fence_after();
      named_bar_sync(kNbSoftmax, kSmThreads);
      if (hc == 0 && tq == 0) {
#pragma unroll
        for (int w2 = 0; w2 < 2; ++w2) {
          const int hd = w2 ? hB : hA;
          if (hd >= NH) continue;
          const float mh = w2 ? mB : mA;
          const float lh = s_lsum[hd] + s_lsum[64 + hd];
          const int hh = hg * NH + hd;
          if (row < 0) {
            const float ms = p.attn_sink[hh] * kLog2e;
            const float M = fmaxf(mh, ms);
            float f = 0.f;
            if (M != -INFINITY && ms != INFINITY) {
              const float a = ex2_approx(mh - M);
              f = a / (lh * a + ex2_approx(ms - M));
            }
            s_fac[hd] = f;
          } else {
            if (rank == 0) p.part_ml[(size_t)row * H + hh] = make_float2(mh, lh);
            s_fac[hd] = 1.f;
          }
        }
      }
      named_bar_sync(kNbSoftmax, kSmThreads);
      const int b = hc;  // warps 4b..4b+3 write O^T block b (rows 128b..128b+127 of this half)
      if (row < 0) {
        // bf16 output: O^T read with the 16x256b shape (thread t: rows
        // d = t/4 and t/4 + 8 of a 16-row band, head pairs 8*rep + 2*(t%4),
        // +1), scaled, packed and transposed by stmatrix into two
        // [NH heads][64 d] 128-byte-swizzled boxes in the idle P buffers,
        // which two TMA stores copy to out.
        uint8_t* stg = smem + C::kOffP + b * (NH * 256);
        constexpr int kCH = NH < 32 ? NH : 32;  // heads (TMEM columns) per chunk
#pragma unroll
        for (int h0 = 0; h0 < NH; h0 += kCH) {
          float fac[kCH / 4];  // this thread's heads h0 + 8*rep + 2*tq, +1
#pragma unroll
          for (int rep = 0; rep < kCH / 8; ++rep) {
            fac[2 * rep] = s_fac[h0 + 8 * rep + 2 * tq];
            fac[2 * rep + 1] = s_fac[h0 + 8 * rep + 2 * tq + 1];
          }
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const uint32_t taddr = tmem + ((uint32_t)(q4 * 32 + 16 * half) << 16) + C::kOCol + b * NH + h0;
            uint32_t r[kCH / 2];
            if constexpr (kCH == 32) tmem_ld_16x256b_x4(taddr, r);
            else tmem_ld_16x256b_x2(taddr, r);
            tmem_wait_ld();
            // "+ 0.f" turns -0 into +0 when the factor is 0 (sink = +inf)
            uint32_t pk[kCH / 4];
#pragma unroll
            for (int rep = 0; rep < kCH / 8; ++rep) {
#pragma unroll
              for (int dg = 0; dg < 2; ++dg) {
                __nv_bfloat162 v2 = __floats2bfloat162_rn(
                    __uint_as_float(r[4 * rep + 2 * dg]) * fac[2 * rep] + 0.f,
                    __uint_as_float(r[4 * rep + 2 * dg + 1]) * fac[2 * rep + 1] + 0.f);
                pk[2 * rep + dg] = *reinterpret_cast<uint32_t*>(&v2);
              }
            }
            const int m = lane >> 3, j = lane & 7;
            const int dl = q4 * 32 + 16 * half + 8 * (m & 1);  // block-local d of the 8 columns
            const int box = dl >> 6, chunk = (dl & 63) >> 3;
#pragma unroll
            for (int rep0 = 0; rep0 < kCH / 8; rep0 += 2) {
              const int h = h0 + 8 * (rep0 + (m >> 1)) + j;
              const uint32_t addr = smem_addr(stg) + box * (NH * 128) + h * 128 + ((chunk ^ (h & 7)) << 4);
              stmatrix_x4_trans(addr, pk[2 * rep0], pk[2 * rep0 + 1], pk[2 * rep0 + 2], pk[2 * rep0 + 3]);
            }
          }
        }
        fence_proxy_async_smem();
        named_bar_sync(kNbBlock0 + b, 128);
        if (q4 == 0 && lane == 0) {
          const int x = (int)rank * kHalf + b * 128;
          tma_store_2d(&tmap_out, x, t * H + hg * NH, smem_addr(stg));
          tma_store_2d(&tmap_out, x + 64, t * H + hg * NH, smem_addr(stg) + NH * 128);
          bulk_commit();
          bulk_wait_read0();  // the staging area (a P buffer) may be rewritten
        }
        named_bar_sync(kNbBlock0 + b, 128);
      } else {
        const int d = (int)rank * kHalf + b * 128 + q4 * 32 + lane;
#pragma unroll
        for (int c = 0; c < NH / 16; ++c) {
          uint32_t ov[16];
          tmem_ld16(tmem + lane_base + C::kOCol + b * NH + c * 16, ov);
          tmem_wait_ld();
          float* o = p.part_o + ((size_t)row * H + hg * NH + c * 16) * kD + d;
#pragma unroll
          for (int e = 0; e < 16; ++e) o[(size_t)e * kD] = __uint_as_float(ov[e]);
        }
      }
      tc_fence_before();
      named_bar_sync(kNbSoftmax, kSmThreads);  // s_fac / s_lsum are rewritten by the next unit
      if (lane == 0) mbar_arrive(bar(kBarOEmpty));
    }
    if (warp == 0 || warp == 4) {
      if (lane == 0) bulk_wait0();  // every output store has landed before the CTA exits
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kQkWarp) tmem_dealloc(tmem, C::kTmemCols);
  cluster_sync_all();  // the partner no longer writes here or arrives on these barriers
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

// 2-D bf16 tensor [rows][512] with 64 x box_rows boxes, 128-byte swizzle
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows,
              CUtensorMapL2promotion promo) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)kD, rows};
  cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, promo,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int NH>
cudaLaunchConfig_t pair_config(int pairs, cudaStream_t st, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = PCfg<NH>::kSmem;
  cfg.stream = st;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

template <int NH>
cudaError_t prepare_nh(int* pairs) {
  *pairs = 0;
  cudaError_t e = cudaFuncSetAttribute(decode_pair_kernel<NH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       PCfg<NH>::kSmem);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pair_config<NH>(1, nullptr, attr);
  cfg.numAttrs = 0;  // the cluster shape is compiled in (__cluster_dims__)
  int n = 0;
  e = cudaOccupancyMaxActiveClusters(&n, decode_pair_kernel<NH>, &cfg);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();  // not fatal: the one-CTA kernel is used instead
    return e;
  }
  *pairs = n;
  return cudaSuccess;
}

template <int NH>
cudaError_t launch_nh(const void* q, const void* kv, const int32_t* kv_indices,
                      const float* attn_sink, float scale, int N, int H, void* out, void* ws,
                      const WsLayout& L, const LaunchPlan& lp, cudaStream_t st) {
  CUtensorMap tq, tout;
  if (!make_map(&tq, q, (uint64_t)N * H, NH, CU_TENSOR_MAP_L2_PROMOTION_L2_128B) ||
      !make_map(&tout, out, (uint64_t)N * H, NH, CU_TENSOR_MAP_L2_PROMOTION_NONE))
    return cudaErrorInvalidValue;
  char* base = static_cast<char*>(ws);
  Params p;
  p.kv = static_cast<const __nv_bfloat16*>(kv);
  p.kv_indices = kv_indices;
  p.attn_sink = attn_sink;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.hdr = reinterpret_cast<WsHeader*>(base);
  p.units = reinterpret_cast<const int4*>(base + L.units_off);
  p.part_ml = reinterpret_cast<float2*>(base + L.ml_off);
  p.part_o = reinterpret_cast<float*>(base + L.o_off);
  p.qk_scale_log2 = scale * kLog2e;
  p.H = H;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pair_config<NH>(lp.grid, st, attr);
  return cudaLaunchKernelEx(&cfg, decode_pair_kernel<NH>, tq, tout, p);
}

}  // namespace

size_t pair_smem_bytes(int nh) {
  switch (nh) {
    case 16: return PCfg<16>::kSmem;
    case 32: return PCfg<32>::kSmem;
    case 64: return PCfg<64>::kSmem;
    default: return 0;
  }
}

cudaError_t pair_prepare(int nh, int* pairs) {
  switch (nh) {
    case 16: return prepare_nh<16>(pairs);
    case 32: return prepare_nh<32>(pairs);
    case 64: return prepare_nh<64>(pairs);
    default: *pairs = 0; return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode_pair(const void* q, const void* kv, const int32_t* kv_indices,
                               const float* attn_sink, float softmax_scale, int N, int H, int D,
                               void* out, void* ws, const WsLayout& L, const LaunchPlan& lp,
                               cudaStream_t st) {
  if (D != kD || lp.grid < 1) return cudaErrorInvalidValue;
  switch (lp.nh) {
    case 16: return launch_nh<16>(q, kv, kv_indices, attn_sink, softmax_scale, N, H, out, ws, L, lp, st);
    case 32: return launch_nh<32>(q, kv, kv_indices, attn_sink, softmax_scale, N, H, out, ws, L, lp, st);
    case 64: return launch_nh<64>(q, kv, kv_indices, attn_sink, softmax_scale, N, H, out, ws, L, lp, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace sda
