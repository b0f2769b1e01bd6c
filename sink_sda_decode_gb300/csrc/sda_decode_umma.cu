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
//  * One persistent CTA per SM owns a contiguous run of work units: a unit
//    is a piece of one token's slot list for NH <= 64 heads (H = 128 uses
//    two CTAs per token, which read the same rows at about the same time,
//    the second mostly from L2).  All heads of a unit share each gathered KV
//    row, so a row is read from memory once per CTA.
//  * Warps 8..23 load KV tiles of 64 slots: warp v copies rows 4v .. 4v+3
//    straight from global to a 128-byte-swizzled shared-memory stage with
//    16-byte cp.async, one half of D per commit group, each half as soon as
//    the PV MMAs that last read it are done (2 stages, 3 for NH = 16); the
//    rows of the tile two ahead are brought into L2 with bulk prefetches.
//    (FP8 pool: two groups of 8 warps on alternate tiles dequantise E4M3
//    codes in registers into the same bf16 tile.)  TMA tile::gather4, which
//    fetches 128 bytes of four rows per instruction, topped out near a third
//    of HBM bandwidth on this GPU.
//  * Warps 24 and 26 issue the QK MMAs (tcgen05, M = 64 padded heads, N = 64
//    slots), warp 24 the first half of D into S_a and warp 26 the second
//    into S_b, so that their MMAs overlap in the tensor pipe; warp 24 also
//    loads q of each unit with tiled TMA.  Softmax thread 0 issues
//    O^T += V^T P^T  (M = 128 rows of D, N = NH heads, K = 64 slots) into a
//    TMEM accumulator right after the barrier at which every softmax warp
//    has written the tile's P; the same shared tile is K (K-major operand)
//    and V (MN-major operand).  Warps 25 and 27 only fill out their
//    warpgroup.
//  * Warps 0..7 read S_a + S_b from TMEM (warps q and q + 4 share lane
//    quadrant q and take slots 0..31 and 32..63), run the online softmax,
//    write P (bf16) to shared memory, rescale O^T in TMEM only when a
//    head's running max grows by more than 8 (2^8 headroom, so p <= 256),
//    and finally normalise with the sink and write out through stmatrix +
//    TMA stores (or, for a piece of a split token, write the unnormalised
//    partial for the combine kernel).
//  * Registers are redistributed with setmaxnreg (softmax warps grow, the
//    loader and MMA warpgroups shrink); every mbarrier wait is bounded (2 s),
//    and on timeout the kernel raises the workspace error word, drains its
//    own copies and returns.
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
constexpr int kPanelKV = kTileN * 128;     // bytes of one KV panel
constexpr int kKVBytes = kPanels * kPanelKV;   // 64 KB per stage
constexpr int kMaxStages = 3;
constexpr int kSmWarps = 8;                // warps 0..7: softmax / epilogue (warps q, q+4 share TMEM quadrant q)
constexpr int kLoaderWarp0 = 8;            // warps 8..23: KV row loaders, two groups of 8
constexpr int kLoaderWarps = 8;            // warps per loader group (group g loads tiles of parity g)
constexpr int kLoaderGroups = 2;
constexpr int kMmaWarp = 24;               // warp 24: QK issuer (first half of D) + q loads
// warps 25 and 27 only fill out the MMA warpgroup (softmax thread 0 issues the PV MMAs)
constexpr int kMmaWarpB = 26;              // warp 26: QK issuer (second half of D)
// 28 warps (27 idle) = 7 warpgroups; registers are split by setmaxnreg:
// softmax warpgroups 0-1 grow to kSmRegs, loader warpgroups 2-5 and the MMA
// warpgroup 6 shrink.  The split must fit the launch allocation of
// kThreads x kLaunchRegs (checked on the host before the first launch).
constexpr int kThreads = 896;
constexpr int kLaunchRegs = 72;            // 65536 / 896, rounded down to a multiple of 8
template <bool FP8>
struct RegSplit {  // the FP8 loaders dequantise in registers, so they get more
  static constexpr int kSm = 96;
  static constexpr int kLoader = FP8 ? 64 : 56;
  static constexpr int kMma = FP8 ? 56 : 72;
  static_assert(kSmWarps * 32 * kSm + kLoaderGroups * kLoaderWarps * 32 * kLoader + 4 * 32 * kMma <=
                    kThreads * kLaunchRegs,
                "register split exceeds the launch allocation");
};
constexpr int kSoftmaxThreads = kSmWarps * 32;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

enum Bar : int {
  kBarQFull = 0,
  kBarQEmpty,
  kBarKVFull0,                                // + 2 * stage + half (columns [256 half, +256))
  kBarPVDone0 = kBarKVFull0 + 2 * kMaxStages,  // + 2 * stage + half (PV blocks 2 half, 2 half + 1 done)
  kBarSFull0 = kBarPVDone0 + 2 * kMaxStages,
  kBarSFull1,
  kBarSEmpty0,
  kBarSEmpty1,
  kBarDrain,
  kBarDrainPv,
  kBarDrainQb,
  kNumBars
};

__host__ __device__ constexpr int kv_full(int s, int h) { return kBarKVFull0 + 2 * s + h; }
__host__ __device__ constexpr int pv_done(int s, int h) { return kBarPVDone0 + 2 * s + h; }

template <int NH>
struct Cfg {
  // q panels are packed NH rows apart; the QK MMA reads 64 rows per panel,
  // so for NH < 64 rows NH..63 of a panel are whatever follows (the next
  // panels, then the first KV stage): valid shared memory whose products
  // land in TMEM lanes that nothing reads.  The space this saves at NH = 16
  // buys a third KV stage.
  static constexpr int kStages = NH <= 16 ? 3 : 2;
  static constexpr int kPanelQ = NH * 128;
  static constexpr int kQBytes = kPanels * kPanelQ;
  static constexpr int kPBytes = NH * 128;  // P: NH rows x 64 slots bf16
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = kQBytes;
  static constexpr int kOffP = kOffKV + kStages * kKVBytes;
  // second output staging area (the first is the two P buffers): the TMA
  // stores of one 128-row block of D read one area while the next block is
  // written into the other
  static constexpr int kOffStage2 = kOffP + kStages * kPBytes;
  static constexpr int kOffBar = kOffStage2 + NH * 256;
  static constexpr int kOffMisc = kOffBar + 256;  // kNumBars <= 32
  // misc: tmem base (4), abort flag (4), pad, then per-head float arrays:
  // l-sum [2 halves][64]; alpha aliases its first half (used only inside a
  // unit's tiles) and fac its second (each thread reads its head's l-sums
  // before it writes that head's fac); half-tile maxima [2 tiles][2][64]
  static constexpr int kOffLSum = kOffMisc + 16;
  static constexpr int kOffAlpha = kOffLSum;
  static constexpr int kOffFac = kOffLSum + 4 * 64;
  static constexpr int kOffHMax = kOffLSum + 4 * 128;
  static constexpr int kSmemUsed = kOffHMax + 4 * 256;
  static constexpr int kSmem = kSmemUsed + 1024;  // slack for 1024-byte alignment
  static constexpr int kOCol = 128;  // O^T block b at columns [128 + b*NH, +NH)
  static constexpr int kSbCol = kOCol + 4 * NH;  // S_b buffers (second half of D) after O^T
  static constexpr int kTmemCols = (kSbCol + 128) <= 256 ? 256 : 512;
  static_assert(kSbCol + 128 <= 512, "TMEM columns");
  static constexpr uint32_t kIdescQK = idesc_bf16_f32(64, 64, false, false);
  static constexpr uint32_t kIdescPV = idesc_bf16_f32(128, NH, true, false);
  static_assert(kOffP % 1024 == 0 && kPBytes % 1024 == 0, "swizzle atoms need 1 KB alignment");
  static_assert(kOffKV % 1024 == 0 && kPanelQ % 1024 == 0, "swizzle atoms need 1 KB alignment");
  static_assert((kPanels - 1) * kPanelQ + kQRows * 128 <= kOffBar, "padded QK A operand inside smem");
  static_assert(kStages <= kMaxStages, "barrier rings");
  static_assert(kNumBars * 8 <= kOffMisc - kOffBar, "mbarrier area");
  static_assert(kSmem <= 232448, "shared memory budget");
};

struct Params {
  const __nv_bfloat16* q;
  const __nv_bfloat16* kv;  // bf16 pool, or (FP8 kernels) the E4M3 codes [P, D] as bytes
  const float* kv_scale;    // FP8 kernels: per-row dequantisation scale [P]
  const int32_t* kv_indices;
  const float* attn_sink;
  __nv_bfloat16* out;
  WsHeader* hdr;
  const int4* units;
  const int* cta_start;  // CTA b's units are units[cta_start[b] .. cta_start[b + 1])
  float2* part_ml;
  float* part_o;
  float qk_scale_log2;
  int H;
  uint64_t wait_timeout_ns;  // bound of every pipeline wait (2 s unless a test shortens it)
  int withhold_arrive;       // test only: CTA 0's first loader warp skips one arrive
};

// Where a bounded wait reports a timeout, and after how long.
struct WaitCtx {
  volatile int* abort_flag;  // shared: set once any role of the CTA gave up
  WsHeader* hdr;             // global error word (1 = a wait timed out)
  uint64_t timeout_ns;
};

// Bounded wait.  Returns false (and raises the abort flags) on timeout; once
// any role has aborted, every later wait returns false at once, so all roles
// run to the end of their loops quickly and the CTA exits.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const WaitCtx& wc) {
  if (mbar_try_wait(bar, parity)) return true;
  if (*wc.abort_flag) return false;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (*wc.abort_flag) return false;
      if (globaltimer_ns() - t0 > wc.timeout_ns) {
        *wc.abort_flag = 1;
        atomicExch(&wc.hdr->error, 1);
        return false;
      }
    }
  }
}

// Wait used only while draining copies / MMAs this CTA started: bounded by
// the timeout, but not cut short by the abort flag.
__device__ __forceinline__ void drain_bar(uint32_t bar, uint32_t parity, const WaitCtx& wc) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > wc.timeout_ns) {
      atomicExch(&wc.hdr->error, 1);
      return;
    }
  }
}

// Walks the tiles of the units a CTA owns (its contiguous run of the unit
// list), in the same order in every role; units without slots are skipped.
struct TileCursor {
  const int4* units;
  int n_units;
  int k;       // unit of the CTA's run
  int4 u;      // current unit
  int ntiles;  // tiles of the current unit
  int i;       // tile within the unit
  int g;       // tiles seen before this one (all units)
  int nu;      // units with slots seen before this one
  bool valid;
  __device__ __forceinline__ int len() const { return u.z; }
  __device__ __forceinline__ void seek() {
    for (;; ++k) {
      if (k >= n_units) {
        valid = false;
        return;
      }
      u = units[k];
      if (u.z > 0) {
        ntiles = (u.z + kTileN - 1) / kTileN;
        i = 0;
        valid = true;
        return;
      }
    }
  }
  __device__ __forceinline__ void init(const int4* us, int n) {
    units = us;
    n_units = n;
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

template <int NH, bool FP8>
__global__ void __launch_bounds__(kThreads, 1)
decode_umma_kernel(const __grid_constant__ CUtensorMap tmap_q,
                   const __grid_constant__ CUtensorMap tmap_out, const Params p) {
  using C = Cfg<NH>;
  constexpr int KS = C::kStages;  // KV stages: tile g lives in stage g % KS
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
  float* s_lsum = reinterpret_cast<float*>(smem + C::kOffLSum);
  float* s_hmax = reinterpret_cast<float*>(smem + C::kOffHMax);
  auto bar = [&](int i) { return sBar + 8u * (uint32_t)i; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(bar(kBarQFull), 1);
    mbar_init(bar(kBarQEmpty), 2);  // both QK issuers' commits
    for (int i = 0; i < 2 * C::kStages; ++i) {
      mbar_init(bar(kBarKVFull0 + i), kLoaderGroups * kLoaderWarps);
      mbar_init(bar(kBarPVDone0 + i), 1);
    }
    mbar_init(bar(kBarSFull0), 2);  // S_a and S_b
    mbar_init(bar(kBarSFull1), 2);
    mbar_init(bar(kBarSEmpty0), kSmWarps);
    mbar_init(bar(kBarSEmpty1), kSmWarps);
    mbar_init(bar(kBarDrain), 1);
    mbar_init(bar(kBarDrainPv), 1);
    mbar_init(bar(kBarDrainQb), 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmap_q);
    tma_prefetch_desc(&tmap_out);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_addr(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // everything above overlaps the previous kernel (PDL); global memory only below
  pdl_wait();
  pdl_trigger();
  const int4* const my_units = p.units + p.cta_start[blockIdx.x];
  const int n_units = p.cta_start[blockIdx.x + 1] - p.cta_start[blockIdx.x];
  const int H = p.H;
  const WaitCtx wc{abort_flag, p.hdr, p.wait_timeout_ns};

  if (warp >= kLoaderWarp0 && warp < kLoaderWarp0 + kLoaderGroups * kLoaderWarps) {
    // ===================================================== KV row loaders
    // All 16 loader warps share every 64-slot tile: warp v copies rows
    // [4v, 4v+4).  The rows of the tile two ahead are brought into L2 with one
    // bulk prefetch per row, so that their loads wait on L2, not on DRAM.
    setmaxnreg_dec<RegSplit<FP8>::kLoader>();
    const uint4* kv4 = reinterpret_cast<const uint4*>(p.kv);
    auto prefetch_rows = [&](int slot_of_lane) {
      constexpr uint32_t kRowBytes = FP8 ? kD : kD * 2;
      if (slot_of_lane >= 0) {
        bulk_prefetch_l2(reinterpret_cast<const uint8_t*>(p.kv) + (size_t)slot_of_lane * kRowBytes, kRowBytes);
        if constexpr (FP8) bulk_prefetch_l2(p.kv_scale + (slot_of_lane & ~3), 16);  // the row's scale
      }
    };
    bool ok = true;
    if constexpr (FP8) {
      // E4M3 pool: all 16 loader warps share every tile, warp v rows [4v, 4v+4)
      // (as for the bf16 pool).  Lane l reads bytes [8l, 8l+8) of each half of
      // a row's 512 codes (one 8-byte load per row and half, both halves in
      // flight before the stage is free) and lanes 0..3 their rows' scales one
      // tile early; the codes are dequantised (code * scale, rounded to bf16)
      // into the same swizzled bf16 tile as the bf16 pool's rows, half by half.
      constexpr int kRows = kTileN / (kLoaderGroups * kLoaderWarps);  // 4 rows per warp
      const int v = warp - kLoaderWarp0;
      const uint8_t* kv8 = reinterpret_cast<const uint8_t*>(p.kv);
      auto slot_of = [&](const TileCursor& x) {  // lanes 0..3: slot of row 4v + lane of tile x, else -1
        const int n = min(kTileN, x.len() - x.i * kTileN);
        const int r = v * kRows + lane;
        return (lane < kRows && r < n) ? __ldg(p.kv_indices + x.u.y + x.i * kTileN + r) : -1;
      };
      TileCursor cu;  // the current tile
      cu.init(my_units, n_units);
      TileCursor nx = cu;  // the next tile
      if (nx.valid) nx.next();
      TileCursor n2 = nx;  // the one after: its slots are read a tile early, its rows prefetched
      if (n2.valid) n2.next();
      int sl0 = cu.valid ? slot_of(cu) : -1;
      int sl1 = nx.valid ? slot_of(nx) : -1;
      float sc0 = (lane < kRows && sl0 >= 0) ? __ldg(p.kv_scale + sl0) : 0.f;
      if (sl1 >= 0) prefetch_rows(sl1);
      for (int g = 0; cu.valid && ok; ++g) {
        const int s = g % KS;  // KV stage
        const int sl2 = n2.valid ? slot_of(n2) : -1;
        int slot_r[kRows];
        float sc_r[kRows];
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
          slot_r[r] = __shfl_sync(0xffffffffu, sl0, r);
          sc_r[r] = __shfl_sync(0xffffffffu, sc0, r);
        }
        // a tail row of a partial tile is zeros (its p is forced to 0)
        uint2 w[2][kRows];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
          for (int r = 0; r < kRows; ++r)
            w[hh][r] = slot_r[r] >= 0
                           ? __ldcg(reinterpret_cast<const uint2*>(kv8 + (size_t)slot_r[r] * kD) + 32 * hh + lane)
                           : make_uint2(0, 0);
        const float sc1 = (lane < kRows && sl1 >= 0) ? __ldg(p.kv_scale + sl1) : 0.f;  // next tile's scales
        uint8_t* stage = smem + C::kOffKV + s * kKVBytes;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          if (g >= KS) {  // the tile KS back in this stage
            if (lane == 0) ok = wait_bar(bar(pv_done(s, hh)), ((g / KS) - 1) & 1, wc);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
          }
          // 16-byte chunk q = 32*hh + lane of each row: panel q/8, chunk q%8;
          // row 4v + r sits at row (4v + r) % 8 of 8-row swizzle atom (4v + r) / 8
          const int q = hh * 32 + lane, k = q & 7;
          uint8_t* atom = stage + (q >> 3) * kPanelKV + (v >> 1) * 1024;
#pragma unroll
          for (int r = 0; r < kRows; ++r) {
            const int r8 = 4 * (v & 1) + r;
            const uint2 c8 = w[hh][r];
            const float sr = sc_r[r];
            *reinterpret_cast<uint4*>(atom + r8 * 128 + ((k ^ r8) << 4)) =
                make_uint4(e4m3x2_to_bf16x2_scaled(c8.x & 0xffffu, sr),
                           e4m3x2_to_bf16x2_scaled(c8.x >> 16, sr),
                           e4m3x2_to_bf16x2_scaled(c8.y & 0xffffu, sr),
                           e4m3x2_to_bf16x2_scaled(c8.y >> 16, sr));
          }
          fence_proxy_async_smem();  // generic-proxy stores -> read by the tensor cores
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(kv_full(s, hh)));
        }
        prefetch_rows(sl2);  // rows (and scales) of tile g + 2 into L2
        cu = nx;
        nx = n2;
        if (n2.valid) n2.next();
        sl0 = sl1;
        sl1 = sl2;
        sc0 = sc1;
      }
    } else {
    // bf16 pool: all 16 loader warps share every tile, warp v (0..15) rows
    // [4v, 4v+4).  Rows go straight from global to shared memory with
    // 16-byte cp.async (no register round trip, no separate shared stores).
    // Each half of D of the warp's rows is one commit group, issued as soon
    // as the PV MMAs that last read that half of the stage are done; the
    // warp then waits for its own copies, fences them to the async proxy
    // (the tensor cores read the stage through it) and arrives, half by half.
    constexpr int kRows = kTileN / (kLoaderGroups * kLoaderWarps);  // 4 rows per warp
    const int v = warp - kLoaderWarp0;
    auto slot_of = [&](const TileCursor& x) {  // lanes 0..3: slot of row 4v + lane of tile x, else -1
      const int n = min(kTileN, x.len() - x.i * kTileN);
      const int r = v * kRows + lane;
      return (lane < kRows && r < n) ? __ldg(p.kv_indices + x.u.y + x.i * kTileN + r) : -1;
    };
    TileCursor cu;  // the current tile
    cu.init(my_units, n_units);
    TileCursor nx = cu;  // the next tile
    if (nx.valid) nx.next();
    TileCursor n2 = nx;  // the one after: its slots are read a tile early, its rows prefetched
    if (n2.valid) n2.next();
    int sl0 = cu.valid ? slot_of(cu) : -1;
    int sl1 = nx.valid ? slot_of(nx) : -1;
    if (sl1 >= 0) prefetch_rows(sl1);
    for (int g = 0; cu.valid && ok; ++g) {
      const int s = g % KS;  // KV stage
      const int sl2 = n2.valid ? slot_of(n2) : -1;
      const uint32_t stage = sKV + s * kKVBytes;
      int slot_r[kRows];  // slots of this warp's rows (-1: past the tile's end)
#pragma unroll
      for (int r = 0; r < kRows; ++r) slot_r[r] = __shfl_sync(0xffffffffu, sl0, r);
      int issued = 0;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        if (g >= KS) {  // the tile KS back in this stage
          if (lane == 0) ok = wait_bar(bar(pv_done(s, hh)), ((g / KS) - 1) & 1, wc);
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;
        }
        // 16-byte chunk q = 32*hh + lane of each row: panel q/8, chunk q%8;
        // row 4v + r sits at row (4v + r) % 8 of 8-row swizzle atom (4v + r) / 8
        // of every panel.  A tail row of a partial tile is zero-filled (its p
        // is forced to 0).
        const int q = hh * 32 + lane, k = q & 7;
        const uint32_t atom = stage + (q >> 3) * kPanelKV + (v >> 1) * 1024;
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
          const int slot = slot_r[r], r8 = 4 * (v & 1) + r;
          const uint4* src = slot >= 0 ? kv4 + (size_t)slot * (kD / 8) + q : kv4;
          cp_async16(atom + r8 * 128 + ((k ^ r8) << 4), src, slot >= 0 ? 16u : 0u);
        }
        cp_async_commit();
        ++issued;
      }
      if (issued == 2) {
        cp_async_wait_group<1>();  // first half landed
        fence_proxy_async_smem();
        __syncwarp();
        // (a test can make CTA 0's first loader warp withhold this arrive
        // once, so that the QK issuer's bounded wait runs out)
        const bool withhold = p.withhold_arrive && blockIdx.x == 0 && v == 0 && g == 0;
        if (lane == 0 && !withhold) mbar_arrive(bar(kv_full(s, 0)));
      }
      cp_async_wait_group<0>();
      if (issued == 2) {
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kv_full(s, 1)));
      }
      prefetch_rows(sl2);  // rows of tile g + 2 into L2
      cu = nx;
      nx = n2;
      if (n2.valid) n2.next();
      sl0 = sl1;
      sl1 = sl2;
    }
    }
  } else if (warp >= kMmaWarp) {
    if constexpr (RegSplit<FP8>::kMma < kLaunchRegs) setmaxnreg_dec<RegSplit<FP8>::kMma>();  // the whole warpgroup (warp 27 idles)
    if (warp == kMmaWarp || warp == kMmaWarpB) {
    // ===================================================== MMA issuers
    // Two threads issue the QK MMAs; one thread's MMAs run one after the
    // other, but MMAs of different threads overlap in the tensor pipe, so
    // splitting the work keeps it busy: warps 24 and 26, lane 0, compute
    // S = Q K^T of every tile, K split in two: warp 24 the columns [0, 256)
    // of D into S_a, warp 26 the columns [256, 512) into S_b (the softmax
    // adds the two), each as soon as its half of the tile has landed and the
    // S buffer is free; warp 24 also loads q of the next unit (tiled TMA) once
    // both halves of this unit's last QK have read q.  (The PV MMAs are
    // issued by softmax thread 0 right after the barrier at which every
    // softmax warp has written the tile's P.)  Each thread's commits track
    // only its own MMAs.  Each has a single next event at any time, so it
    // sleeps in the mbarrier wait (hardware suspend) instead of spinning,
    // leaving the issue slots to the other warps.
    if (lane == 0) {
      const int qh = warp == kMmaWarpB ? 1 : 0;  // QK: half of D (of the K dimension)
      TileCursor cq;
      cq.init(my_units, n_units);
      int q_issued = 0;
      bool ok = true;
      if (qh == 0 && cq.valid) {  // q of the first unit
        mbar_arrive_expect_tx(bar(kBarQFull), NH * 128 * kPanels);
        const int qrow = cq.u.x * H + unit_head_group(cq.u.w) * NH;
#pragma unroll
        for (int c = 0; c < kPanels; ++c) tma_load_2d(sQ + c * C::kPanelQ, &tmap_q, c * 64, qrow, bar(kBarQFull));
        q_issued = 1;
      }
      while (cq.valid && ok) {
        const int g = cq.g, s = g & 1, ks = g % KS;  // S buffer, KV stage
        {
          if (g >= 2) ok = wait_bar(bar(kBarSEmpty0 + s), ((g >> 1) - 1) & 1, wc);
          if (ok && cq.i == 0) ok = wait_bar(bar(kBarQFull), cq.nu & 1, wc);
          if (ok) ok = wait_bar(bar(kv_full(ks, qh)), (g / KS) & 1, wc);
          if (!ok) break;
          tc_fence_after();
          const uint32_t kvs = sKV + ks * kKVBytes;
          // descriptors of the first K step; the others only move the start address
          const uint64_t a0 = sdesc_sw128(sQ, 16, 1024), b0 = sdesc_sw128(kvs, 16, 1024);
          const uint32_t sacc = tmem + (qh ? C::kSbCol : 0) + s * 64;
#pragma unroll
          for (int c = 4 * qh; c < 4 * qh + 4; ++c) {  // panels of this half of D
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t a = sdesc_advance(a0, c * C::kPanelQ + kk * 32);
              const uint64_t bd = sdesc_advance(b0, c * kPanelKV + kk * 32);
              mma_bf16(sacc, a, bd, C::kIdescQK, (c != 4 * qh || kk) ? 1u : 0u);
            }
          }
          mma_commit(bar(kBarSFull0 + s));
          const bool last = cq.i == cq.ntiles - 1;
          const int nu = cq.nu;
          if (last) mma_commit(bar(kBarQEmpty));
          cq.next();
          if (qh == 0 && last && cq.valid) {
            // q of the next unit once this unit's QKs (both halves) have read q
            ok = wait_bar(bar(kBarQEmpty), nu & 1, wc);
            if (!ok) break;
            mbar_arrive_expect_tx(bar(kBarQFull), NH * 128 * kPanels);
            const int qrow = cq.u.x * H + unit_head_group(cq.u.w) * NH;
#pragma unroll
            for (int c = 0; c < kPanels; ++c) tma_load_2d(sQ + c * C::kPanelQ, &tmap_q, c * 64, qrow, bar(kBarQFull));
            q_issued = cq.nu + 1;
          }
        }
      }
      // drain this thread's MMAs (and the last q copy) before TMEM and smem go away
      const int drain = qh ? kBarDrainQb : kBarDrain;
      mma_commit(bar(drain));
      drain_bar(bar(drain), 0, wc);
      if (qh == 0 && q_issued >= 1) drain_bar(bar(kBarQFull), (q_issued - 1) & 1, wc);
    }
    __syncwarp();
    }
  } else if (warp < kSmWarps) {
    setmaxnreg_inc<RegSplit<FP8>::kSm>();
    // ===================================================== softmax + epilogue
    // Warp w reads TMEM lane quadrant q = w % 4 and slots [32hc, 32hc + 32) of
    // each tile, hc = w / 4, with the 16x256b shape: thread t holds heads
    // hA = 16q + t/4 and hB = hA + 8 (the M = 64 accumulator keeps row r in
    // lane 32*(r/16) + r%16) for the 8 slots 32hc + 8rep + 2(t%4) + {0,1},
    // rep = 0..3, as the sum of the two K halves S_a + S_b.
    //
    // Weights are taken against a per-head running reference m (log2
    // units): p = 2^(score * scale * log2 e - m).  On a unit's first tile m
    // is the tile's exact per-head maximum (two quad shuffles and an
    // exchange with warp w ^ 4).  On later tiles the weights are computed
    // against the current m straight away, and only when a scaled score
    // exceeds m by more than the threshold (2^8 headroom, so p <= 256 in
    // bf16) do the eight warps take the exact path: the tile's maxima, a
    // raised m, O^T rescaled in TMEM and the tile's weights recomputed.  So
    // a tile after the first needs one block-wide vote and no exchange, and
    // the weights are those of a running maximum raised lazily.
    const int q4 = warp & 3, hc = warp >> 2;
    const int st = threadIdx.x;  // 0..255
    const int tq = lane & 3;
    const int hA = q4 * 16 + (lane >> 2), hB = hA + 8;
    const bool vA = hA < NH, vB = hB < NH;
    const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
    const float sc = p.qk_scale_log2;
    // Control flow here is identical in the eight warps (it depends only on
    // the unit list and on block-wide votes), so every named barrier is
    // reached by all of them even after a wait timed out: a timed-out wait
    // only leaves garbage in the outputs and the error word raised.
    int g = 0;
    for (int k = 0; k < n_units; ++k) {
      const int4 u = my_units[k];
      const int t = u.x, len = u.z, hg = unit_head_group(u.w), row = unit_part_row(u.w);
      if (len <= 0) {
        // padded token: out = 0 for its NH heads (contiguous NH*D bf16)
        uint4* o = reinterpret_cast<uint4*>(p.out + ((size_t)t * H + hg * NH) * kD);
        for (int e = st; e < NH * kD / 8; e += kSoftmaxThreads) o[e] = make_uint4(0, 0, 0, 0);
        continue;
      }
      const int ntiles = (len + kTileN - 1) / kTileN;
      float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;  // l: this thread's share
      // the sink logits are only needed in the epilogue: load them now
      const float sinkA = (row < 0 && vA && tq == 0 && hc == 0) ? __ldg(p.attn_sink + hg * NH + hA) : 0.f;
      const float sinkB = (row < 0 && vB && tq == 0 && hc == 0) ? __ldg(p.attn_sink + hg * NH + hB) : 0.f;
      for (int i = 0; i < ntiles; ++i, ++g) {
        const int s = g & 1;
        const int n = min(kTileN, len - i * kTileN);
        wait_bar(bar(kBarSFull0 + s), (g >> 1) & 1, wc);
        tc_fence_after();
        float x[16];  // raw scores of this thread's 16 (head, slot) pairs: S_a + S_b
        {
          uint32_t sa[16], sb[16];  // both halves in flight before one wait
          tmem_ld_16x256b_x4(tmem + lane_base + s * 64 + 32 * hc, sa);
          tmem_ld_16x256b_x4(tmem + lane_base + C::kSbCol + s * 64 + 32 * hc, sb);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e) x[e] = __uint_as_float(sa[e]) + __uint_as_float(sb[e]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kBarSEmpty0 + s));  // S buffer s may be overwritten
        uint32_t valid = 0;  // bit e: element e is a slot of the list (not past the tile's end)
#pragma unroll
        for (int rep = 0; rep < 4; ++rep) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const int j = 32 * hc + 8 * rep + 2 * tq + (kk & 1);
            valid |= (j < n ? 1u : 0u) << (4 * rep + kk);
          }
        }
        // P buffer s is free once the PV of tile g-2 is done
        if (g >= 2) {
          if (lane == 0) wait_bar(bar(pv_done((g - 2) % KS, 1)), ((g - 2) / KS) & 1, wc);
          __syncwarp();
        }
        // p = 2^(x*scale - m) in bf16 into rows hA, hB of P (K-major, 128-byte
        // swizzle: 16-byte chunk c of 8 slots at (c ^ (h & 7)) * 16).  The
        // 16x256b load left this thread's weights in the layout of stmatrix
        // fragments (row = head t/4 of an 8-head group, columns = slot pair
        // 2(t%4) of an 8-slot chunk), so each warp stores its 16 heads x 32
        // slots with two stmatrix.x4 (matrix i = chunk 4hc + i; lane 8i + j
        // addresses head row j).  Returns whether a weight exceeded the
        // headroom.  The denominator sums the same bf16 weights the PV MMA
        // multiplies, so rounding p perturbs the weights of an exact weighted
        // average but biases nothing.
        const uint32_t prow = sP + s * C::kPBytes + (2 * q4) * 1024 + (lane & 7) * 128 +
                              ((((4 * hc) + (lane >> 3)) ^ (lane & 7)) << 4);
        float sA, sB;
        auto weights = [&]() {
          bool over = false;
          sA = 0.f;
          sB = 0.f;
          uint32_t pa[4], pb[4];
#pragma unroll
          for (int rep = 0; rep < 4; ++rep) {
            float e[4];
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const bool ok_e = (valid >> (4 * rep + kk)) & 1u;
              const float arg = fmaf(x[4 * rep + kk], sc, -((kk < 2) ? mA : mB));
              over = over || (ok_e && arg > kRescaleThreshold);
              e[kk] = ok_e ? ex2_approx(arg) : 0.f;
            }
            __nv_bfloat162 va = __floats2bfloat162_rn(e[0], e[1]), vb = __floats2bfloat162_rn(e[2], e[3]);
            const float2 fa = __bfloat1622float2(va), fb = __bfloat1622float2(vb);
            sA += fa.x + fa.y;
            sB += fb.x + fb.y;
            pa[rep] = *reinterpret_cast<uint32_t*>(&va);
            pb[rep] = *reinterpret_cast<uint32_t*>(&vb);
          }
          if (vA) {  // warp-uniform (vA == vB)
            stmatrix_x4(prow, pa[0], pa[1], pa[2], pa[3]);
            stmatrix_x4(prow + 1024, pb[0], pb[1], pb[2], pb[3]);
          }
          return over;
        };
        // exact path on a unit's first tile (block-uniform), else by vote (an
        // invalid head's weights are never stored, so it casts no vote)
        bool exact = i == 0;
        if (!exact) {
          const bool over = weights() && vA;
          fence_proxy_async_smem();  // this thread's P stores -> read by the tensor cores
          exact = named_bar_or(1, kSoftmaxThreads, over);
        }
        if (exact) {
          // exact path: the tile's largest scaled score per head
          float eA = -INFINITY, eB = -INFINITY;
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            if ((valid >> e) & 1u) {
              if ((e & 3) < 2) eA = fmaxf(eA, x[e] * sc);
              else eB = fmaxf(eB, x[e] * sc);
            }
          }
#pragma unroll
          for (int o = 1; o <= 2; o <<= 1) {
            eA = fmaxf(eA, __shfl_xor_sync(0xffffffffu, eA, o));
            eB = fmaxf(eB, __shfl_xor_sync(0xffffffffu, eB, o));
          }
          {  // combine with the other half of the tile (warp w ^ 4)
            float* hm = s_hmax + (g & 1) * 128;
            if (tq == 0) {
              hm[hc * 64 + hA] = eA;
              hm[hc * 64 + hB] = eB;
            }
            named_bar_sync(2 + q4, 64);
            eA = fmaxf(eA, hm[(hc ^ 1) * 64 + hA]);
            eB = fmaxf(eB, hm[(hc ^ 1) * 64 + hB]);
          }
          float alphaA = 1.f, alphaB = 1.f;
          if (vA && eA > mA + kRescaleThreshold) {
            alphaA = ex2_approx(mA - eA);  // 0 when m was -inf
            lA *= alphaA;
            mA = eA;
          }
          if (vB && eB > mB + kRescaleThreshold) {
            alphaB = ex2_approx(mB - eB);
            lB *= alphaB;
            mB = eB;
          }
          weights();  // against the raised reference (the scores die here)
          fence_proxy_async_smem();
          if (i > 0) {
            // O^T already holds this unit's earlier tiles: scale its head columns
            if (tq == 0 && hc == 0) {
              if (vA) s_alpha[hA] = alphaA;
              if (vB) s_alpha[hB] = alphaB;
            }
            named_bar_sync(1, kSoftmaxThreads);
            // O^T must be quiescent: wait for the PV of tile g-1
            if (lane == 0) wait_bar(bar(pv_done((g - 1) % KS, 1)), ((g - 1) / KS) & 1, wc);
            __syncwarp();
            tc_fence_after();
            // this warp's lanes of O^T blocks 2hc, 2hc + 1
#pragma unroll
            for (int b = 2 * hc; b < 2 * hc + 2; ++b) {
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
          }
          // every warp's P (and rescaled O^T) is written; s_alpha is rewritten next time
          tc_fence_before();
          named_bar_sync(1, kSoftmaxThreads);
        }
        lA += sA;
        lB += sB;
        // O^T += V^T P^T of this tile, issued by one thread now that the last
        // barrier (the vote, or the exact path's) has seen every warp's P: a
        // commit after blocks 1 and 3 releases each half of the KV stage (the
        // second also frees the P buffer and marks O^T complete).  The same
        // shared tile is K (K-major) for QK and V (MN-major) here.
        if (threadIdx.x == 0) {
          tc_fence_after();
          const int ks = g % KS;
          const uint32_t kvs = sKV + ks * kKVBytes;
          const uint32_t ps = sP + s * C::kPBytes;
          const uint64_t a0 = sdesc_sw128(kvs, kPanelKV, 1024), b0 = sdesc_sw128(ps, 16, 1024);
#pragma unroll
          for (int b = 0; b < 4; ++b) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              // A = V^T block b: rows d in [128b, 128b+128) = panels 2b, 2b+1 (MN-major);
              //     K = slots [16kk, 16kk+16) = row groups 2kk, 2kk+1
              const uint64_t a = sdesc_advance(a0, (2 * b) * kPanelKV + kk * 2048);
              // B = P^T: N = NH heads (rows), K = 16 slots at byte offset 32kk (K-major)
              const uint64_t bd = sdesc_advance(b0, kk * 32);
              mma_bf16(tmem + C::kOCol + b * NH, a, bd, C::kIdescPV, (i == 0 && kk == 0) ? 0u : 1u);
            }
            if (b & 1) mma_commit(bar(pv_done(ks, b >> 1)));
          }
        }
        __syncwarp();
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
      if (lane == 0) wait_bar(bar(pv_done(gl % KS, 1)), (gl / KS) & 1, wc);
      __syncwarp();
      tc_fence_after();
      named_bar_sync(1, kSoftmaxThreads);
      if (tq == 0 && hc == 0) {
#pragma unroll
        for (int w2 = 0; w2 < 2; ++w2) {
          const int hd = w2 ? hB : hA;
          const float mh = w2 ? mB : mA;
          if (hd >= NH) continue;
          const float lh = s_lsum[hd] + s_lsum[64 + hd];  // read before fac[hd] overwrites s_lsum[64 + hd]
          const int hh = hg * NH + hd;
          float f = 1.f;
          if (row < 0) {
            const float ms = (w2 ? sinkB : sinkA) * kLog2e;
            const float M = fmaxf(mh, ms);
            f = 0.f;
            if (M != -INFINITY && ms != INFINITY) {
              const float a = ex2_approx(mh - M);
              f = a / (lh * a + ex2_approx(ms - M));
            }
          } else {
            p.part_ml[(size_t)row * H + hh] = make_float2(mh, lh);
          }
          s_fac[hd] = f;
        }
      }
      named_bar_sync(1, kSoftmaxThreads);
      if (row < 0) {
        // bf16 output: warps 4hc..4hc+3 write O^T blocks 2hc and 2hc + 1
        // (rows 256hc..256hc+255 of D) through staging area hc.  O^T is read
        // with the 16x256b shape (thread t: rows d = t/4 and t/4 + 8 of a
        // 16-row band, head pairs 8*rep + 2*(t%4), +1) in chunks of 32 heads,
        // scaled, packed to bf16 pairs and written transposed with stmatrix as
        // two [NH heads][64 d] boxes in the 128-byte-swizzled layout (no bank
        // conflicts), which two TMA stores copy to out.
        uint8_t* stg = smem + (hc ? C::kOffStage2 : C::kOffP);  // 2 boxes of NH x 128 B
        constexpr int kCH = NH < 32 ? NH : 32;  // heads per chunk
#pragma unroll 1
        for (int b = 2 * hc; b < 2 * hc + 2; ++b) {
          if (b & 1) {
            // the stores of block b - 1 have read the staging area
            if (q4 == 0 && lane == 0) bulk_wait_read0();
            named_bar_sync(6 + hc, 128);
          }
#pragma unroll
          for (int h0 = 0; h0 < NH; h0 += kCH) {
            float fac[kCH / 4];  // this thread's heads h0 + 8*rep + 2*tq, +1
#pragma unroll
            for (int rep = 0; rep < kCH / 8; ++rep) {
              fac[2 * rep] = s_fac[h0 + 8 * rep + 2 * tq];
              fac[2 * rep + 1] = s_fac[h0 + 8 * rep + 2 * tq + 1];
            }
            // both 16-row bands of the quadrant in flight before one wait
            uint32_t rr[2][kCH / 2];
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              const uint32_t taddr = tmem + ((uint32_t)(q4 * 32 + 16 * half) << 16) + C::kOCol + b * NH + h0;
              if constexpr (kCH == 32) tmem_ld_16x256b_x4(taddr, rr[half]);
              else tmem_ld_16x256b_x2(taddr, rr[half]);
            }
            tmem_wait_ld();
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              const uint32_t (&r)[kCH / 2] = rr[half];
              // "+ 0.f" turns -0 into +0 when the factor is 0 (sink = +inf)
              uint32_t pk[kCH / 4];  // [rep][row d or d+8]
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
              // matrix m of a stmatrix.x4 = (rep0 + m/2, d group m%2); lane
              // 8m + j addresses row j (head h0 + 8*rep + j) of matrix m
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
          named_bar_sync(6 + hc, 128);
          if (q4 == 0 && lane == 0) {
            tma_store_2d(&tmap_out, b * 128, t * H + hg * NH, smem_addr(stg));
            tma_store_2d(&tmap_out, b * 128 + 64, t * H + hg * NH, smem_addr(stg) + NH * 128);
            bulk_commit();
          }
        }
        // the staging areas (one is the P buffers) are free again before
        // this unit's epilogue ends
        if (q4 == 0 && lane == 0) bulk_wait_read0();
      } else {
#pragma unroll 1
        for (int b = 2 * hc; b < 2 * hc + 2; ++b) {
          const int d = b * 128 + q4 * 32 + lane;
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
      }
      // s_fac / s_lsum are rewritten, and O^T is overwritten by the next unit's
      // first PV (issued by thread 0 after a later barrier)
      tc_fence_before();
      named_bar_sync(1, kSoftmaxThreads);
    }
    if (threadIdx.x == 0) {  // every PV MMA done before TMEM and shared memory go away
      mma_commit(bar(kBarDrainPv));
      drain_bar(bar(kBarDrainPv), 0, wc);
    }
    if (q4 == 0 && lane == 0) bulk_wait0();  // every output store has landed before the CTA exits
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, C::kTmemCols);
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
                 uint32_t box_rows, CUtensorMapL2promotion promo,
                 CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, promo,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int NH, bool FP8>
cudaError_t launch_nh(const void* q, const void* kv, const float* kv_scale, int64_t total_pages,
                      const int32_t* kv_indices, const float* attn_sink, float scale, int N, int H,
                      void* out, void* ws, const WsLayout& L, const LaunchPlan& lp, cudaStream_t st) {
  (void)total_pages;
  CUtensorMap tq, tout;
  if (!make_map_2d(&tq, q, kD, (uint64_t)N * H, 64, NH, CU_TENSOR_MAP_L2_PROMOTION_L2_128B) ||
      !make_map_2d(&tout, out, kD, (uint64_t)N * H, 64, NH, CU_TENSOR_MAP_L2_PROMOTION_NONE))
    return cudaErrorInvalidValue;
  char* base = static_cast<char*>(ws);
  Params p;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.kv = static_cast<const __nv_bfloat16*>(kv);
  p.kv_scale = kv_scale;
  p.kv_indices = kv_indices;
  p.attn_sink = attn_sink;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.hdr = reinterpret_cast<WsHeader*>(base);
  p.units = reinterpret_cast<const int4*>(base + L.units_off);
  p.cta_start = reinterpret_cast<const int*>(base + L.cta_off);
  p.part_ml = reinterpret_cast<float2*>(base + L.ml_off);
  p.part_o = reinterpret_cast<float*>(base + L.o_off);
  p.qk_scale_log2 = scale * kLog2e;
  p.H = H;
  const WaitFault wf = current_wait_fault();
  p.wait_timeout_ns = wf.timeout_ns;
  p.withhold_arrive = wf.withhold;
  return launch_pdl(decode_umma_kernel<NH, FP8>, dim3(lp.grid), dim3(kThreads), (size_t)Cfg<NH>::kSmem,
                    st, tq, tout, p);
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

// The warp roles resize their registers with setmaxnreg, and an increase
// waits until the others have released enough of the CTA's launch
// allocation: never launch a build whose allocation is smaller than the split
// assumes (the increase would wait forever).
template <int NH, bool FP8>
cudaError_t prepare_variant() {
  cudaError_t e = cudaFuncSetAttribute(decode_umma_kernel<NH, FP8>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<NH>::kSmem);
  if (e != cudaSuccess) return e;
  cudaFuncAttributes a;
  e = cudaFuncGetAttributes(&a, decode_umma_kernel<NH, FP8>);
  if (e != cudaSuccess) return e;
  if (a.numRegs < kLaunchRegs || a.maxThreadsPerBlock < kThreads) return cudaErrorInvalidConfiguration;
  return cudaSuccess;
}

template <int NH>
cudaError_t prepare_nh() {
  cudaError_t e = prepare_variant<NH, false>();
  if (e == cudaSuccess) e = prepare_variant<NH, true>();
  return e;
}

cudaError_t umma_prepare(int nh) {
  switch (nh) {
    case 16: return prepare_nh<16>();
    case 32: return prepare_nh<32>();
    case 64: return prepare_nh<64>();
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode_umma(const void* q, const void* kv, const float* kv_scale,
                               int64_t total_pages, const int32_t* kv_indices,
                               const float* attn_sink, float softmax_scale, int N, int H, int D,
                               void* out, void* ws, const WsLayout& L, const LaunchPlan& lp,
                               cudaStream_t st) {
  if (D != kD) return cudaErrorInvalidValue;
  const bool fp8 = kv_scale != nullptr;
#define SDA_LAUNCH(NHV)                                                                          \
  return fp8 ? launch_nh<NHV, true>(q, kv, kv_scale, total_pages, kv_indices, attn_sink,          \
                                    softmax_scale, N, H, out, ws, L, lp, st)                      \
             : launch_nh<NHV, false>(q, kv, nullptr, total_pages, kv_indices, attn_sink,         \
                                     softmax_scale, N, H, out, ws, L, lp, st)
  switch (lp.nh) {
    case 16: SDA_LAUNCH(16);
    case 32: SDA_LAUNCH(32);
    case 64: SDA_LAUNCH(64);
    default: return cudaErrorInvalidValue;
  }
#undef SDA_LAUNCH
}

}  // namespace sda
