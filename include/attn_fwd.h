/*
 * attn_fwd.h -- C ABI of the exact attention forward pass for GB300 (sm_103a).
 *
 * Operation.  For every batch b, query head h and query row i:
 *     O[b,h,i,:] = sum_j P_ij V[b,g(h),j,:],   P_ij = exp(s_ij - LSE_i),
 *     s_ij       = scale * <Q[b,h,i,:], K[b,g(h),j,:]>   over the allowed keys j,
 *     LSE[b,h,i] = ln sum_j exp(s_ij)                    (natural log, scale included),
 * with g(h) = h / (Hq / Hkv) (grouped-query attention: consecutive query heads
 * share a key/value head).  This is softmax attention with its closed-form
 * log-sum-exp normaliser (page "AdaSplash-2: Faster Differentiable Sparse
 * Attention", technical summary section 1), computed fused in the
 * FlashAttention manner (same section: fused operations kept in on-chip
 * memory), so the Sq x Sk score matrix never reaches HBM.  It is the attention
 * forward pass whose hand-written single-file CUDA kernels the article "L'agent
 * a questions depasse l'agent a outils : 113% contre 50% de la vitesse de
 * FlashAttention-3" reports for Hopper and Blackwell (section "Ce que cela a
 * donne").
 *
 * Masks (`causal`):
 *     0  every key is allowed;
 *     1  bottom-right aligned: key j is allowed for row i iff j <= i + (Sk - Sq)
 *        (for Sq == Sk this is the usual top-left causal mask);
 *     2  top-left aligned: key j is allowed for row i iff j <= i.
 *     A row with no allowed key gets O = 0 and LSE = -inf.
 *
 * Layout (all contiguous, row-major, device memory):
 *     q [B][Hq][Sq][D] bf16     k, v [B][Hkv][Sk][D] bf16
 *     o [B][Hq][Sq][D] bf16     lse  [B][Hq][Sq] fp32
 * D must be 64 or 128; Hq must be a multiple of Hkv; scale must be finite and
 * positive (1/sqrt(D) is the usual value); every pointer must be 16-byte
 * aligned.  o and lse must not overlap q, k, v or each other.
 *
 * Ownership and execution.  The caller owns every buffer.  attn_fwd allocates
 * no device memory; it enqueues one kernel on `stream` (0 = legacy default
 * stream) and returns without synchronising, so errors raised while the kernel
 * runs surface on the stream (or through attn_fwd_debug_status).  Inputs are
 * not modified.  Calls are re-entrant; the one-time initialisation (driver
 * entry point, per-device capability check and kernel attributes) is guarded.
 *
 * Work order.  A launch's work items (256 query rows of one head) are handed to
 * the CTAs heaviest first with heads fastest.  In the dense forward (attn_fwd,
 * and attn_fwd_splitkv with one split), when K and V of all kv heads exceed the
 * L2 cache (long contexts, chunked prefill over them), the items of each kv head
 * are handed out together instead, heaviest first within the kv head, so that K
 * and V tiles are not read again from HBM wave after wave.  The order never
 * changes the results: every output element is computed the same way in either
 * order.  The environment variable ATTN_FWD_ITEM_ORDER=heads or =grouped, read
 * at each call, forces one order.
 *
 * Concurrency.  Each forward launch (attn_fwd and every variant below) claims
 * its work items from one of a set of device counters and returns that counter
 * to zero as it finishes.  Launches made directly take 64 counters in turn;
 * launches recorded into a CUDA graph (stream capture) take another 4096 in turn
 * and keep theirs for every replay.  So: at most 64 direct launches may be in
 * flight on one device at once (on different streams); a direct launch never
 * shares a counter with a recorded one; and launches recorded 4096 or more
 * captures apart may share one, so graphs holding them must not run at the same
 * time.  Two launches that did share a counter while running would silently
 * skip or repeat work items.
 *
 * Precision.  bf16 inputs; both products accumulate in fp32 on the tensor
 * cores; softmax in fp32 with exp2.  The P.V product runs in fp16: P is rounded
 * to fp16 (nearest-even) and the normaliser sums those same rounded values, and
 * each V tile is converted to fp16 inside the kernel (exact for magnitudes in
 * [2^-14, 65504]; smaller ones round to fp16's subnormal grid, an absolute
 * error below 2^-25).  V entries beyond 65504 in magnitude are outside the
 * supported range: they are clamped to +-65504 in the P.V product, so the rows
 * that give such a key weight come out wrong (but finite) while every other
 * row is unaffected.  O is rounded to bf16 (nearest-even) once, at the end.
 */
#ifndef ATTN_FWD_H
#define ATTN_FWD_H

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes (0 = success). */
#define ATTN_OK 0
#define ATTN_ERR_INVALID_ARG 1        /* a size < 0, Hq or Hkv < 1, D not 64/128, Hq % Hkv, causal not 0..2,
                                         scale not finite and > 0, overlapping outputs, or a size beyond
                                         the 32-bit index range */
#define ATTN_ERR_NULL_PTR 2           /* a required pointer is NULL */
#define ATTN_ERR_MISALIGNED 3         /* a pointer is not 16-byte aligned */
#define ATTN_ERR_UNSUPPORTED_DEVICE 4 /* the current device is not compute capability 10.3 (sm_103a) */
#define ATTN_ERR_CUDA 5               /* a CUDA runtime call failed; see attn_fwd_strerror(ATTN_ERR_CUDA) */
#define ATTN_ERR_DEVICE_TIMEOUT 6     /* a kernel wait ran out of time and the kernel unwound (debug status) */
#define ATTN_ERR_TENSOR_MAP 7         /* the driver rejected a TMA tensor map for these pointers and sizes */

/*
 * Enqueue the attention forward pass on `stream`.
 * Returns ATTN_OK or one of the codes above.  Argument checks run on the host
 * before any device work; nothing is launched when a check fails.  With
 * B == 0 or Sq == 0 there is nothing to compute and the call returns ATTN_OK
 * without launching.  Sk == 0 is valid: every row is fully masked.
 */
int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int Sq,
             int Sk, int D, int causal, float scale, cudaStream_t stream);

/*
 * Split-key forward: the same operation and result as attn_fwd, for shapes
 * with too few (batch, head, 256-row query block) work items to fill the GPU
 * (a short query chunk against a long key/value cache).  The visible key tiles
 * of every work item are cut into n_splits contiguous ranges processed as
 * separate items; each range writes its partial O (fp32, normalised within the
 * range) and partial LSE into `workspace`, and a second kernel merges them:
 *     LSE = ln sum_r exp(LSE_r),   O = sum_r exp(LSE_r - LSE) O_r.
 * This is the log-sum-exp identity of the closed-form softmax normaliser (page
 * "AdaSplash-2: Faster Differentiable Sparse Attention", technical summary
 * section 1) applied to a partition of the keys.
 *
 * workspace: caller-owned device memory, 16-byte aligned, at least
 * attn_fwd_splitkv_workspace_size(B, Hq, Sq, D, n_splits) bytes, not overlapping
 * any input or output; its contents are overwritten.  1 <= n_splits <= 256.
 * Two kernels are enqueued on `stream` (one when n_splits == 1: the plain
 * forward, which gives the same values, and the workspace is left untouched);
 * nothing is allocated.  Other arguments,
 * layouts and status codes as attn_fwd (ATTN_ERR_INVALID_ARG also for a
 * too-small workspace).
 */
int attn_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                     int Sq, int Sk, int D, int causal, float scale, int n_splits, void* workspace,
                     size_t workspace_bytes, cudaStream_t stream);

/* Workspace bytes attn_fwd_splitkv needs: n_splits * B*Hq*Sq * (D + 1) * 4 plus
   alignment; 0 for invalid sizes.  Host only, no CUDA call. */
size_t attn_fwd_splitkv_workspace_size(int B, int Hq, int Sq, int D, int n_splits);

/* A split count for the current device, from a cost model of the launch on
   GB300: the work items of every split count run in waves over the SMs (so a
   split that fills the last wave can pay even when the items already outnumber
   the SMs), against the merge's extra traffic; at least four 128-key tiles per
   range, and 1 unless a split is predicted to gain at least 3 %. */
int attn_fwd_splitkv_suggest(int B, int Hq, int Sq, int Sk, int D, int causal);

/*
 * attn_fwd_splitkv without a workspace argument, for callers that cannot
 * allocate device memory: code that is handed only its input and output
 * buffers (an operator or plugin interface with no workspace) and must not
 * call cudaMalloc itself, because a raw cudaMalloc can synchronise the device
 * and goes around the memory manager that owns the GPU's memory.  (There is no
 * counterpart on the pages; this is a calling convention of this library.)
 *
 * Same operation, arguments, result and status codes as attn_fwd_splitkv.  The
 * partials live in a fixed 32 MiB device array inside the library instead of a
 * workspace: calls whose n_splits * B*Hq*Sq * (D + 1) * 4 bytes (plus up to 255
 * bytes of alignment) exceed 32 MiB are rejected with ATTN_ERR_INVALID_ARG
 * before any device work.  Nothing is allocated: every GPU that loads the
 * library holds the 32 MiB until the process exits.  The first call in each
 * CUDA context looks up the array's device address there (a host-side query;
 * again after a cudaDeviceReset, which ends the context), so make that first
 * call before any stream capture.  All calls share the one array and
 * each call overwrites what it needs (nothing has to start at zero), so calls
 * that overlap on the GPU -- on different streams, or on the same device from
 * different threads without ordering -- race and must be serialised by the caller.
 */
int attn_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                             int Hkv, int Sq, int Sk, int D, int causal, float scale, int n_splits,
                             cudaStream_t stream);

/*
 * Block-sparse forward: attn_fwd restricted to the (query block, key block)
 * pairs a bit-packed mask marks.  Key j is visible to row i iff the causal rule
 * allows it AND the mask bit of (query block i / ATTN_MASK_BLOCK, key block
 * j / ATTN_MASK_BLOCK) is set; key blocks whose bit is clear are never loaded.
 * This is the bit-packed block masking of page "AdaSplash-2: Faster
 * Differentiable Sparse Attention" (technical summary section 2: one bit per
 * block of the attention matrix, 32 blocks per 32-bit word, the output pass
 * visiting only the marked blocks) applied to exact softmax attention.  A row
 * with no visible key gets O = 0 and LSE = -inf.
 *
 * block_mask: device memory, 4-byte aligned, uint32 words laid out
 *     [B][mask_heads][ceil(Sq / ATTN_MASK_BLOCK)][W],  W = ceil(ceil(Sk / ATTN_MASK_BLOCK) / 32),
 * bit (kb % 32) of word (kb / 32) marking key block kb; bits past the last key
 * block are ignored.  mask_heads is 1 (one mask for every head) or Hq.  The mask
 * is read by the kernel and must not change until it has finished; it must not
 * overlap o or lse.  Other arguments, layouts and status codes as attn_fwd
 * (ATTN_ERR_INVALID_ARG also for a mask_heads that is neither 1 nor Hq).  One
 * kernel is enqueued on `stream`; nothing is allocated.
 */
#define ATTN_MASK_BLOCK 128
int attn_fwd_blocksparse(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                         int Sq, int Sk, int D, int causal, float scale, const uint32_t* block_mask, int mask_heads,
                         cudaStream_t stream);

/* Number of uint32 words of a block mask for these sizes (layout above); 0 for
   invalid sizes.  Host only, no CUDA call. */
size_t attn_fwd_block_mask_words(int B, int mask_heads, int Sq, int Sk);

/*
 * Ordered forward: attn_fwd with the key tiles of every 256-row query block
 * visited in a caller-given order.  This is the ordered-skipping kernel of page
 * "CoSA: Accelerating Long-Context Inference via Proxy-Kernel Co-Designed Sparse
 * Attention" (a proxy hands the kernel a priority list and the kernel reads the
 * blocks in that order, so the most important ones come first) on the exact
 * path: nothing is skipped that the list contains, so with a list holding every
 * key tile the result is attention itself, the visiting order changing only the
 * rounding of the sums.  The block of query rows [256 u, 256 u + 256) visits, in
 * list order, every entry e of its row with 0 <= e < (its causal key-tile bound);
 * entries outside that range are passed over.  A row that leaves a tile out makes
 * that tile's keys invisible to the block (block-sparse attention); a tile listed
 * twice is counted twice, so rows should list each tile at most once.
 *
 * tile_order: device memory, 4-byte aligned, int32 entries laid out
 *     [B][order_heads][ceil(Sq / ATTN_ORDER_ROWS)][ceil(Sk / ATTN_ORDER_KEYS)],
 * entry values being key-tile indices (tile kb holds keys [128 kb, 128 kb + 128)).
 * order_heads is 1 (one order for every head) or Hq.  The order is read by the
 * kernel and must not change until it has finished; it must not overlap o or
 * lse.  Other arguments, layouts and status codes as attn_fwd
 * (ATTN_ERR_INVALID_ARG also for an order_heads that is neither 1 nor Hq).  One
 * kernel is enqueued on `stream`; nothing is allocated.
 */
#define ATTN_ORDER_ROWS 256
#define ATTN_ORDER_KEYS 128
int attn_fwd_ordered(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int Sq,
                     int Sk, int D, int causal, float scale, const int32_t* tile_order, int order_heads,
                     cudaStream_t stream);

/* Number of int32 entries of a tile order for these sizes (layout above); 0 for
   invalid sizes.  Host only, no CUDA call. */
size_t attn_fwd_tile_order_entries(int B, int order_heads, int Sq, int Sk);

/* Text for a status code.  For ATTN_ERR_CUDA it names the CUDA error of the
   calling thread's most recent failing call. */
const char* attn_fwd_strerror(int status);

/* Library version: major * 10000 + minor * 100 + patch. */
int attn_fwd_version(void);

/*
 * Synchronise `stream`, then read and clear the library's device status word
 * for the current device.  Every wait inside the kernel is bounded (a few
 * seconds); a wait that runs out records where it gave up and the kernel
 * unwinds cleanly instead of hanging.  Returns ATTN_OK, ATTN_ERR_DEVICE_TIMEOUT,
 * or ATTN_ERR_CUDA when the synchronisation itself reports an error.
 * `site` (may be NULL) receives the recorded code (0 when none).
 */
int attn_fwd_debug_status(cudaStream_t stream, int* site);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_FWD_H */
