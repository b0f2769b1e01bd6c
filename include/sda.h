/*
 * sda.h -- C ABI of libsda: sparse decode attention with a per-head attention
 * sink over a unified KV pool, for NVIDIA GB300 (sm_103a).
 *
 * The operation is the one documented by the docstring of paged_decode.py,
 * quoted on the sglang PR 28392 summary page ("为 AMD V4 内核添加 ATOM 来源注释",
 * section "关键源码片段"): caller convention, returns and numerics.
 *
 * Conventions shared by every entry point:
 *   - All tensor arguments are raw DEVICE pointers into memory the caller
 *     owns (e.g. torch tensors' data_ptr()).  The library never allocates,
 *     frees or keeps them.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  Every call only enqueues work on that stream: there is no
 *     host synchronisation, no device-to-host read and no allocation, so the
 *     calls can be captured into a CUDA graph.
 *   - Host-side argument checks happen before anything is enqueued; on
 *     failure nothing is enqueued and an error code is returned.
 *     SDA_ERR_CUDA means a launch failed (cudaGetLastError() was not
 *     cudaSuccess); the message is in sda_last_cuda_error().
 *   - Errors found on the device never trap: they are written to status
 *     words that the caller reads when it chooses.
 */
#ifndef SDA_H_
#define SDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum sda_status {
  SDA_OK = 0,
  SDA_ERR_INVALID_ARG = 1, /* null pointer, bad size, misaligned pointer        */
  SDA_ERR_UNSUPPORTED = 2, /* (H, D) outside the supported set                  */
  SDA_ERR_CUDA = 3,        /* a CUDA call or launch failed                       */
  SDA_ERR_WORKSPACE = 4    /* workspace smaller than sda_decode_workspace_size() */
} sda_status;

/* Human-readable name of a status code (static string, never NULL). */
const char* sda_strerror(sda_status status);

/* Text of the last CUDA error seen by this library on the calling thread
 * ("" if none).  Static thread-local storage; never NULL. */
const char* sda_last_cuda_error(void);

/* ABI version of this header (bumped on any signature change). */
int sda_abi_version(void);

/*
 * Bytes of device workspace sda_decode needs for a call with these sizes on
 * the CURRENT device (it depends on the device's SM count, which fixes how
 * long token lists are split across CTAs).  Writes the size to *bytes.
 * total_indices is the length of kv_indices.  Returns SDA_ERR_UNSUPPORTED for
 * an (H, D) that sda_decode rejects, SDA_ERR_CUDA if no device is usable.
 */
sda_status sda_decode_workspace_size(int N, int H, int D, int64_t total_indices, size_t* bytes);

/*
 * Sparse decode attention with an attention sink (paged_decode.py docstring:
 * caller convention, returns, numerics).
 *
 *   q            [N, H, D] bf16, contiguous, 16-byte aligned.
 *   unified_kv   [total_pages, D] bf16, contiguous, 16-byte aligned; one row
 *                (page size 1) is both the key and the value of a slot.
 *                0 < total_pages < 2^31.
 *   kv_indices   [total_indices] int32.  Token t attends over
 *                kv_indices[kv_indptr[t] : kv_indptr[t+1]].  CONTRACT: every
 *                entry inside those slices is a valid slot in
 *                [0, total_pages) -- the kernels do not bounds-check slots
 *                (check with sda_validate_indices when in doubt).
 *   kv_indptr    [N + 1] int32, non-decreasing, within [0, total_indices];
 *                kv_indptr[0] need not be 0.  A padded token has an empty
 *                slice (kv_indptr[t+1] == kv_indptr[t]) and gets out = 0.
 *   attn_sink    [H] fp32: per-head sink logit (natural-log units, not scaled
 *                by softmax_scale); it adds e^sink to the softmax denominator
 *                as a key whose value is zero.  May be -inf (no sink).
 *   softmax_scale  multiplies q.k before the softmax.
 *   out          [N, H, D] bf16 (q's dtype), written with round-to-nearest-
 *                even; must not overlap the inputs.
 *   workspace    device scratch of at least sda_decode_workspace_size()
 *                bytes, 256-byte aligned; its contents need no
 *                initialisation and are overwritten.  Two calls in flight
 *                at the same time must use different workspaces.
 *
 * Supported: D in {64, 128, 256, 512}, 1 <= H <= 256 (D = 512 with
 * H in {16, 32, 64, 128, 192, 256} takes the tensor-core path).
 * N = 0 is a no-op.  Softmax is computed online in the log2 domain in fp32.
 */
sda_status sda_decode(const void* q, const void* unified_kv, int64_t total_pages,
                      const int32_t* kv_indices, int64_t total_indices,
                      const int32_t* kv_indptr, const float* attn_sink, float softmax_scale,
                      int N, int H, int D, void* out, void* workspace, size_t workspace_bytes,
                      void* stream);

/*
 * Workspace bytes sda_decode_fp8 needs for these sizes (as
 * sda_decode_workspace_size, for the FP8-pool kernel).  SDA_ERR_UNSUPPORTED
 * for an (H, D) that sda_decode_fp8 rejects.
 */
sda_status sda_decode_fp8_workspace_size(int N, int H, int D, int64_t total_indices,
                                         size_t* bytes);

/*
 * sda_decode over a pool stored in FP8: the same attention (paged_decode.py
 * docstring: caller convention, returns, numerics) with row s, element d of
 * the pool worth e4m3(kv_fp8[s, d]) * kv_scale[s].  The pages keep unified_kv
 * in bf16 and quantise to FP8 only on the cache-store side (the fused
 * RMSNorm + RoPE + FP8 quantisation + paged SWA store kernel of the sglang
 * PR 25898 summary page, "关键文件"); this entry point is the pool format
 * that halves the gathered bytes: one FP8 E4M3 code per element (sign, 4
 * exponent bits with bias 7, 3 mantissa bits, no infinities, S.1111.111 =
 * NaN) and one fp32 dequantisation scale per row.
 *
 *   kv_fp8       [total_pages, D] E4M3 codes (one byte each), contiguous,
 *                16-byte aligned.
 *   kv_scale     [total_pages] fp32, 4-byte aligned; any finite value
 *                (0 makes the row an all-zero key and value).
 *   other arguments, results, contract and errors as sda_decode; workspace
 *   of at least sda_decode_fp8_workspace_size() bytes.
 *
 * Numerics: each gathered element is dequantised to bf16 (code * scale,
 * rounded to nearest even) in shared memory, then the tensor-core path
 * computes exactly as for a bf16 pool.  With power-of-two scales (as 8-bit
 * exponent block scales are) that product is exact, so the result is as
 * accurate as sda_decode's on the dequantised pool; any other scale rounds
 * each element once more (relative 2^-9).  Supported: D = 512 with H in {16, 32,
 * 64, 128, 192, 256}; other shapes return SDA_ERR_UNSUPPORTED.
 */
sda_status sda_decode_fp8(const void* q, const void* kv_fp8, const float* kv_scale,
                          int64_t total_pages, const int32_t* kv_indices, int64_t total_indices,
                          const int32_t* kv_indptr, const float* attn_sink, float softmax_scale,
                          int N, int H, int D, void* out, void* workspace, size_t workspace_bytes,
                          void* stream);

/*
 * sda_decode without a workspace argument, for callers that cannot allocate
 * device memory: hosts that give an operator only its input and output
 * buffers and forbid it to allocate (e.g. an inference engine that owns all
 * device memory under a fixed budget), or C callers with no device allocator
 * of their own.  The paper has no counterpart; this is a service of this
 * library.
 *
 * Same arguments, results and errors as sda_decode, except the workspace:
 * the scratch memory is a fixed device array of SDA_NOALLOC_SCRATCH_BYTES
 * (16 MiB) inside this library, which every GPU that loads the library holds
 * until the process exits.  The call allocates and frees nothing.
 *   - A call whose sda_decode_workspace_size() exceeds
 *     SDA_NOALLOC_SCRATCH_BYTES returns SDA_ERR_WORKSPACE and enqueues
 *     nothing (e.g. H = 16, D = 512 fits; H >= 64 at D = 512 on a GB300
 *     does not: use sda_decode with a workspace of your own there).
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture begins.
 *   - All calls on a device share the one array and it keeps the last call's
 *     contents.  Nothing in it has to start at zero (every call rewrites what
 *     it reads), but two calls that overlap on the GPU -- on different
 *     streams, or from different threads -- race on it: order them.
 */
#define SDA_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)
sda_status sda_decode_noalloc(const void* q, const void* unified_kv, int64_t total_pages,
                              const int32_t* kv_indices, int64_t total_indices,
                              const int32_t* kv_indptr, const float* attn_sink,
                              float softmax_scale, int N, int H, int D, void* out, void* stream);

/*
 * Which attention kernel sda_decode launches for (H, D) on the current
 * device: *kernel = SDA_KERNEL_SIMT (CUDA cores, any supported shape) or
 * SDA_KERNEL_ONE_CTA (tensor cores, one persistent CTA per SM, each owning an
 * equal share of the batch's KV tiles; D = 512 and H in
 * {16, 32} or a multiple of 64, the default there).  The environment
 * variable SDA_FORCE_VARIANT=simt|umma overrides the choice where the shape
 * allows (for testing).  Errors: SDA_ERR_INVALID_ARG (kernel
 * is NULL), SDA_ERR_UNSUPPORTED, SDA_ERR_CUDA.
 */
#define SDA_KERNEL_SIMT 0
#define SDA_KERNEL_ONE_CTA 1
sda_status sda_decode_kernel(int H, int D, int* kernel);

/*
 * Device-side error word of the last sda_decode that used `workspace`:
 * copies one int32 (0 = fine, nonzero = a pipeline wait timed out and the
 * affected outputs are unspecified) into *device_flag (device memory),
 * ordered on `stream`.
 */
sda_status sda_decode_error_flag(const void* workspace, int32_t* device_flag, void* stream);

/*
 * Timing hook.  When both events are non-NULL, every later sda_decode /
 * sda_decode_fp8 made from the calling host thread records `before` on its
 * stream immediately before its attention kernel and `after` immediately
 * after it, and every later sda_qk_norm_rope_swa_store(_fp8) / sda_topk_slots
 * does the same around its kernel(s), so that the caller can time them alone
 * (cudaEventElapsedTime).  The events are
 * cudaEvent_t handles created and owned by the caller.  NULL, NULL turns the
 * hook off.  No effect on results.
 */
sda_status sda_set_timing_events(void* before, void* after);

/*
 * Test hook for the bounded pipeline waits of the tensor-core kernels (no
 * counterpart on the pages: it exists so that the failure path can be run
 * without faulting anything).  Every later launch of those kernels from any
 * host thread bounds each mbarrier wait by `timeout_ns` (0 = the default of
 * 2 s), and, when withhold_arrive is 1, the first loader warp of CTA 0 skips
 * its arrive on the first half of its first tile, so that the QK issuer's
 * wait runs out: the kernel raises the error word (1), every role drains its
 * own copies and MMAs, and the call completes with unspecified outputs.
 * withhold_arrive must be 0 or 1 (else SDA_ERR_INVALID_ARG).  Reset with
 * (0, 0) before any normal use.
 */
sda_status sda_debug_wait_fault(int withhold_arrive, uint64_t timeout_ns);

/*
 * Index builder (the decode index scatter the docstring calls
 * write_v4_paged_decode_indices; its inputs are not on the page, these are
 * the plainest inputs that produce its two slot formulas).  Per token t:
 *   - state_slot[t] < 0: padded token, empty slice (not an error);
 *   - otherwise swa_len[t] SWA slots, oldest -> newest, ring position
 *     (swa_head[t] - swa_len[t] + 1 + j) mod win, emitted as
 *     state_slot[t] * win + ring;
 *   - then its compressed entries e in [comp_indptr[t], comp_indptr[t+1]),
 *     in input order, emitted as swa_pages + comp_block[e] * k_per_block +
 *     comp_slot[e].
 * kv_indptr [N + 1] receives the prefix sum (kv_indptr[0] = 0) and
 * kv_indices [capacity] the packed slots; entries past kv_indptr[N] are
 * unspecified (the builder uses them as scratch).  All arrays are int32
 * device memory.  A token with a bad field gets an empty slice and sets bits of
 * *status (device int32, overwritten):
 *   1  swa_len outside [0, win]
 *   2  swa_head outside [0, win) while swa_len > 0
 *   4  comp_indptr decreasing or outside [0, comp_total]
 *   8  a compressed entry with block < 0 or slot outside [0, k_per_block)
 *   16 a slot outside its region (state_slot*win + win > swa_pages, or a
 *      compressed slot >= total_pages)
 *   32 the packed lists exceed `capacity`: then every slice is empty
 * So every emitted slot is valid for sda_decode by construction.  The
 * compressed entries are checked in parallel slices of the entry array; a
 * batch that holds bad entries is then re-checked token by token by one CTA
 * (slower, same result).
 * Host errors (SDA_ERR_INVALID_ARG): N < 0, win <= 0, k_per_block <= 0,
 * swa_pages < 0, total_pages outside (0, 2^31), swa_pages > total_pages,
 * capacity < 0 or > 2^31 - 1, a null pointer that would be read.
 */
sda_status sda_build_indices(const int32_t* state_slot, const int32_t* swa_len,
                             const int32_t* swa_head, const int32_t* comp_indptr,
                             const int32_t* comp_block, const int32_t* comp_slot,
                             int64_t comp_total, int N, int win, int k_per_block,
                             int64_t swa_pages, int64_t total_pages, int32_t* kv_indices,
                             int64_t capacity, int32_t* kv_indptr, int32_t* status,
                             void* stream);

/*
 * sda_build_indices followed by sda_decode (or sda_decode_fp8 when kv_scale is
 * not NULL, unified_kv then holding the E4M3 codes), as one call: the same
 * arguments, contracts, outputs and status bits as those two calls made back
 * to back on the stream with total_indices = capacity, with one launch fewer
 * (the decode's work plan runs in the same launch as the builder's scatter).  The
 * workspace is sized by sda_decode_workspace_size (or
 * sda_decode_fp8_workspace_size) with total_indices = capacity.  Lists the
 * builder empties (bad descriptors, or bit 32: over capacity) decode to +0.
 */
sda_status sda_build_decode(const int32_t* state_slot, const int32_t* swa_len,
                            const int32_t* swa_head, const int32_t* comp_indptr,
                            const int32_t* comp_block, const int32_t* comp_slot,
                            int64_t comp_total, int win, int k_per_block, int64_t swa_pages,
                            int32_t* kv_indices, int64_t capacity, int32_t* kv_indptr,
                            int32_t* status, const void* q, const void* unified_kv,
                            const float* kv_scale, int64_t total_pages, const float* attn_sink,
                            float softmax_scale, int N, int H, int D, void* out, void* workspace,
                            size_t workspace_bytes, void* stream);

/*
 * sda_build_decode from HOST buffers: q [N,H,D] bf16, the builder's
 * descriptors (state_slot, swa_len, swa_head [N], comp_indptr [N+1],
 * comp_block, comp_slot [comp_total]) and the outputs out [N,H,D] bf16 and
 * status [1] int32 are page-locked host memory (cudaHostAlloc /
 * cudaMallocHost / torch pin_memory; q and out 16-byte aligned); the pool
 * (unified_kv, kv_scale) and attn_sink stay in device memory.  The call
 * gathers the inputs into `workspace` (device, 256-byte aligned, at least
 * sda_build_decode_host_workspace_size bytes) with one kernel that reads the
 * host memory directly, runs sda_build_decode there (kv_indices and kv_indptr
 * live in the workspace) and writes out and status back to the host with
 * another kernel -- no copy-engine transfer, so the whole step is one
 * sequence of kernels on `stream` (graph-capturable).
 * Batches whose q is 8 MB or more (N*H*D*2 >= 2^23) take another route,
 * because the host link then costs more than the step (about 210 GB/s in and
 * 190 GB/s out on a GB300 with NVLink-C2C): the descriptors and q travel by
 * copy engine on a library-owned inbound stream, in 2..8 token chunks (chunk
 * boundaries depend on N only); the index build runs once for the whole
 * batch on `stream`, then the decode chunk by chunk as each chunk's q lands,
 * and each chunk's out goes back on a library-owned outbound stream as soon
 * as its decode is done, so both link directions and the SMs work at once.
 * `stream` forks to those two streams at the start of the call and joins
 * them at its end (graph-capturable; the two streams and their events are
 * created on the device by the first sda_build_decode_host_workspace_size
 * query or call for such a batch, which must therefore come before any
 * capture; calls from several host threads are serialised while they
 * enqueue).  Each chunk
 * has its own work plan, so the result can differ from the one-call path in
 * the last bf16 bit (both are within the decode's tolerance); status is the
 * whole batch's, as in sda_build_decode.  Asynchronous: the host
 * buffers must stay valid (and keep their page-locking) until the stream has
 * passed this call, and out/status are ready once the stream reaches this
 * point.  SDA_ERR_INVALID_ARG if a host buffer is not page-locked or is
 * misaligned, or on any argument sda_build_decode would reject; those checks
 * all run before anything is enqueued.  Only the start of each host buffer
 * can be checked: the library cannot learn the size of a page-locked
 * allocation, so a host buffer shorter than its stated extent (N*H*D*2 bytes
 * for q and out, 4*N for the per-token descriptors, 4*(N+1) for comp_indptr,
 * 4*comp_total for comp_block / comp_slot) is undefined behaviour: the
 * kernels would read or write past it.
 */
sda_status sda_build_decode_host_workspace_size(int N, int H, int D, int64_t comp_total,
                                                int64_t capacity, int fp8, size_t* bytes);

sda_status sda_build_decode_host(const int32_t* state_slot, const int32_t* swa_len,
                                 const int32_t* swa_head, const int32_t* comp_indptr,
                                 const int32_t* comp_block, const int32_t* comp_slot,
                                 int64_t comp_total, int win, int k_per_block, int64_t swa_pages,
                                 int64_t capacity, const void* q, const void* unified_kv,
                                 const float* kv_scale, int64_t total_pages,
                                 const float* attn_sink, float softmax_scale, int N, int H, int D,
                                 void* out, int32_t* status, void* workspace,
                                 size_t workspace_bytes, void* stream);

/*
 * Checks the docstring's index contract on the device.  status [2] int32
 * device memory receives: status[0] bits 1 = kv_indptr decreasing somewhere,
 * 2 = kv_indptr outside [0, total_indices], 4 = some entry of
 * kv_indices[0 : total_indices] outside [0, total_pages); status[1] = the
 * number of such entries.
 */
sda_status sda_validate_indices(const int32_t* kv_indices, int64_t total_indices,
                                const int32_t* kv_indptr, int N, int64_t total_pages,
                                int32_t* status, void* stream);

/*
 * Top-k selection straight into the compressed slot lists of
 * sda_build_indices.  Source: the sglang attention tag page, entry "DSV4.1
 * 新增索引器内核，重做 Top-K v2 分派" (NaN padding ranks below a legitimate
 * -inf; the page-table transform is a separate step from the selection); the
 * compressed pool entry block_id * K_PER_BLOCK + slot_in_block is the
 * paged_decode.py docstring's (PR 28392 page).
 *
 * Arguments (device pointers):
 *   scores      [N, score_stride] fp32; token t's candidates are positions
 *               p < n_t = lengths[t] (later positions are padding: never read)
 *   lengths     [N] int32; outside [0, score_stride] counts as 0 (bit 1)
 *   block_table [N, bt_stride] int32: position p of token t lies in block
 *               block_table[t][p / k_per_block] at slot p % k_per_block;
 *               bt_stride * k_per_block >= score_stride
 *   k >= 0, k_per_block > 0; comp_block / comp_slot hold `capacity` entries.
 * Per token: the min(k, n_t) best candidates -- larger score first, -0 equal
 * to +0, NaN below -inf (bit 8 if any NaN is a candidate), equal scores by
 * increasing position -- emitted in increasing position as
 * (comp_block, comp_slot) = (block_table[t][p / k_per_block], p % k_per_block);
 * comp_indptr [N + 1] is the prefix sum of min(k, n_t), comp_indptr[0] = 0.
 * *status (device int32, overwritten): bits 1 (bad length), 4 (a kept
 * position has a negative block id, emitted as is), 8 (NaN candidate), 32
 * (the total exceeds capacity: every list is empty).  The outputs are exactly
 * sda_build_indices' comp_indptr / comp_block / comp_slot inputs.  Two
 * launches; graph-capturable; the timing hook brackets both.
 */
sda_status sda_topk_slots(const float* scores, int64_t score_stride, const int32_t* lengths,
                          const int32_t* block_table, int64_t bt_stride, int N, int k,
                          int k_per_block, int32_t* comp_indptr, int32_t* comp_block,
                          int32_t* comp_slot, int64_t capacity, int32_t* status, void* stream);

/*
 * Fused q / kv RMSNorm + RoPE + SWA ring store: the step of a decode layer
 * that fills the pool sda_decode reads.  Source: the sglang PR 25898 summary
 * page ("修复 DSV4 在 AMD GPU 上的运行时崩溃与 JIT 不兼容"), section "关键文件"
 * (fused_qk_norm_rope_store.py: Q per-head RMSNorm, KV RMSNorm, RoPE, FP8
 * quantisation and the paged SWA store in one kernel), section "关键符号"
 * (_batched_rmsnorm, _gptj_rotate, fused_qk_norm_rope_swa_store) and
 * "实现拆解" item 2 (cos_cache / sin_cache); the ring slot state_slot * win +
 * ring is the paged_decode.py docstring's (PR 28392 page).
 *
 * Arguments (device pointers unless noted; all 16-byte aligned except
 * positions, state_slot, status):
 *   q          [N, H, D] bf16, the step's query heads (read)
 *   kv         [N, D] bf16, the step's new latent row per token (key = value)
 *   q_norm_w, kv_norm_w  [D] bf16 RMSNorm weights (q's shared by all heads)
 *   cos_cache, sin_cache [max_pos, rope_dim / 2] fp32, row = position
 *   positions  [N] int32, state_slot [N] int32 (< 0: padded token)
 *   D % 8 == 0, 8 <= D <= 2048; rope_dim % 8 == 0, 0 <= rope_dim <= D;
 *   N * (H + 1) <= 2^30;
 *   eps >= 0 finite; win > 0; 0 <= swa_pages <= total_pages.
 *   q_out      [N, H, D] bf16; may be q itself, must not partly overlap it.
 * Per token t with state_slot[t] >= 0 and 0 <= pos = positions[t] < max_pos,
 * for every row x (the H rows of q[t] with q_norm_w, and kv[t] with kv_norm_w),
 * in fp32:
 *   y_d = x_d / sqrt(mean_d x_d^2 + eps) * w_d
 *   for i < rope_dim/2, d = D - rope_dim + 2i ("GPT-J": adjacent pairs):
 *     (y_d, y_{d+1}) <- (y_d c - y_{d+1} s, y_{d+1} c + y_d s),
 *     c = cos_cache[pos][i], s = sin_cache[pos][i]
 *   q_out[t] = y rounded to nearest even bf16;
 *   the KV row goes to slot = state_slot[t] * win + pos mod win.
 * Padded tokens (and real tokens whose position is outside [0, max_pos)) get
 * q_out = 0 and store nothing.  *status (device int32, overwritten): bit 1 =
 * a real token had a position outside [0, max_pos); bit 2 = a slot fell
 * outside [0, swa_pages) (that row is not stored).  Two tokens with the same
 * slot in one call race (the caller's contract: one new entry per ring slot).
 */
sda_status sda_qk_norm_rope_swa_store(const void* q, const void* kv, const void* q_norm_w,
                                      const void* kv_norm_w, const float* cos_cache,
                                      const float* sin_cache, int max_pos,
                                      const int32_t* positions, const int32_t* state_slot, int N,
                                      int H, int D, int rope_dim, float eps, int win,
                                      int64_t swa_pages, int64_t total_pages, void* q_out,
                                      void* unified_kv, int32_t* status, void* stream);

/*
 * As sda_qk_norm_rope_swa_store, into the FP8 pool of sda_decode_fp8
 * (kv_fp8 [total_pages, D] E4M3 codes, 16-byte aligned; kv_scale
 * [total_pages] fp32): the row's scale is 2^e, e the least integer with
 * 448 * 2^e >= max_d |y_d| (e >= -126; 1 for an all-zero row) -- a power of
 * two, like the UE8M0 scales of block-scaled FP8 -- and code_d = y_d / 2^e
 * rounded to the nearest E4M3 value (ties to even).  The quantised value is
 * computed from the fp32 y, not from its bf16 rounding.
 */
sda_status sda_qk_norm_rope_swa_store_fp8(const void* q, const void* kv, const void* q_norm_w,
                                          const void* kv_norm_w, const float* cos_cache,
                                          const float* sin_cache, int max_pos,
                                          const int32_t* positions, const int32_t* state_slot,
                                          int N, int H, int D, int rope_dim, float eps, int win,
                                          int64_t swa_pages, int64_t total_pages, void* q_out,
                                          void* kv_fp8, float* kv_scale, int32_t* status,
                                          void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SDA_H_ */
