// attn_fwd.cu -- exact attention forward pass for GB300 (sm_103a), fused so the
// Sq x Sk score matrix stays on chip (page "AdaSplash-2: Faster Differentiable
// Sparse Attention", technical summary section 1: FlashAttention's fused,
// on-chip softmax attention with a closed-form log-sum-exp normaliser).
//
// Persistent kernel: one CTA per SM walks a list of work items, each 256 query
// rows (two 128-row Q tiles) of one (batch, query head).  Items are ordered
// heaviest first (most key tiles under a causal mask), heads fastest -- or, in
// the grouped instantiation the host picks when K and V exceed L2, kv head by kv
// head, heaviest first within each; CTA c starts on item c and claims later
// items from a counter as it frees up, so the CTAs end within about one small
// item of each other.  Twelve warps:
//   warps 0-3   softmax for Q tile 0 (one thread per query row), then its epilogue
//   warps 4-7   softmax for Q tile 1, then its epilogue
//   warp  8     TMA producer: the Q tiles of an item, then its K/V tiles through a
//               ring of shared-memory slots guarded by full/empty mbarriers
//   warp  9     tcgen05 issuer: S_t = Q_t K^T into tensor memory (TMEM), and
//               O_t += P_t V with P_t read back from TMEM; owns the TMEM allocation
//   warp  10    idle (it completes the third warpgroup)
//   warp  11    TMA stores of O once the softmax warps have staged it
// Registers are rebalanced per warpgroup after set-up: the softmax warpgroups
// grow to 224 per thread (a whole S row lives in registers), the third shrinks
// to 56; 128*56 + 256*224 equals the 384*168 the block is launched with.
//
// The issuer interleaves the two Q tiles so the tensor cores work on one tile
// while the other tile's softmax runs:
//   S0(0) S1(0) | PV0(j) S0(j+1) PV1(j) S1(j+1) | ...
// and carries on into the next item while the softmax warps run the epilogue of
// the last one: only the first P.V of the next item waits for the epilogue to
// have read O out of TMEM (o_empty), and the next item's Q only waits for the
// last S of this one (q_empty).
// TMEM columns: S0 [0,128)  S1 [128,256)  O0 [256,256+D)  O1 [384,384+D); P_t
// (fp16 pairs) overwrites the last 64 columns of S_t once S_t is in registers,
// so the S of the first 64 keys stays readable until the next S_t.
//
// P.V runs in fp16: P is rounded to fp16 (11 significant bits against bf16's 8,
// which keeps the rounding of P four times smaller) and each V tile is converted
// to fp16 in place in its ring slot before its product, by the softmax warps
// between one tile's hand-off and the next tile's S (exact for |v| in [2^-14,
// 65504]; smaller magnitudes round to fp16's subnormal grid, larger ones are
// clamped to +-65504, so masked keys, whose P is 0, never turn a row non-finite).
//
// Online softmax per row, in log2 units (c = scale * log2 e), with a lazy
// reference value m: a tile's exponentials are taken against the current m,
// and the tile's row max is only computed on a row's first tile (or while it
// has seen no key), where m is set 8 above it, so P starts at most 2^-8 and a
// later key may exceed that first max by up to 2^24 before P leaves fp16's
// range.  When a tile's P mass does pass fp16's largest value 65504 (the rare
// case), m moves up by the power of two that brings the mass below 2^-8 (keys
// 0-63 scale their fp32 P, keys 64-127 redo theirs from S), or, for a mass
// beyond 2^64 or not finite, to 8 above the tile's row max.  Any m gives the
// exact result because O and both normalisers share it.  l sums the
// fp16-rounded P values the tensor cores multiply (taken after P has been handed
// to the MMA), so the final O / l is a convex combination of V rows; a second,
// fp32 sum of the unrounded P gives the LSE.  Causal masking touches only the
// tiles that straddle the diagonal (or the ragged end of K); tiles wholly above
// the diagonal are never loaded.
//
// Every mbarrier wait is bounded: a wait that runs out sets a shared abort
// flag and a device status word, and all roles unwind to the final barrier,
// the issuer drains its MMAs and the producer its copies before TMEM is freed.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <atomic>
#include <mutex>
#include <type_traits>

#include "attn_fwd.h"
#include "host_util.h"
#include "ptx.cuh"

using namespace attn;

namespace {

constexpr int BM = 128;          // query rows per Q tile (MMA M)
constexpr int BN = 128;          // keys per K/V tile
constexpr int QTILES = 2;        // Q tiles per work item
constexpr int ROWS_PER_ITEM = QTILES * BM;
constexpr int kThreads = 384;    // 3 warpgroups
constexpr int kLoadWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kStoreWarp = 11;  // O stores of the epilogue
constexpr uint32_t kRegsLaunch = 168;   // 65536 / 384, what ptxas assigns under the launch bounds
constexpr uint32_t kRegsSoftmax = 224;  // warpgroups 0 and 1
constexpr uint32_t kRegsOther = 56;     // warpgroup 2 (producer, issuer, two idle warps)
static_assert(128 * kRegsOther + 256 * kRegsSoftmax <= kThreads * kRegsLaunch, "register split exceeds the pool");
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kTimeoutNs = 4000000000ull;  // 4 s per wait
constexpr uint64_t kDrainTimeoutNs = 500000000ull;
constexpr float kHeadroom = 8.0f;       // log2 units: m is set this far above a tile's row max
constexpr int kHeadroomBits = 8;
constexpr float kF16Max = 65504.0f;     // largest finite fp16: a tile's P mass above it may overflow
constexpr float kScaleMassLimit = 18446744073709551616.0f;  // 2^64: beyond it a tile is redone from S

// Sites recorded in the device status word when a wait runs out.
constexpr int kSiteProducer = 1;
constexpr int kSiteIssuer = 2;
constexpr int kSiteSoftmax = 3;
constexpr int kSiteEpilogue = 4;

template <int D>
struct Cfg {
  static constexpr int kTileBytes = BN * D * 2;            // one K or V tile; also one Q tile
  static constexpr int kColBlockBytes = BN * 128;          // 64 columns x 128 rows, 128-B swizzled
  static constexpr int kStages = (D == 128) ? 4 : 8;       // K/V ring slots
  static constexpr int kQBytes = QTILES * BM * D * 2;
  static constexpr int kStageBytes = BM * D * 2;           // one Q tile of O in bf16, 128-B swizzled
  static constexpr int kStageBufs = (D == 128) ? 1 : 2;    // O staging buffers (1: the two Q tiles take turns)
  // D = 64: the P.V product is D + 16 columns wide, its last 16 columns multiplying
  // P by a block of ones, so the tensor cores accumulate the rounded-P row sum l
  // next to O (TMEM has room for it only at D = 64).
  static constexpr bool kTensorRowSum = (D == 64);
  static constexpr int kPvN = kTensorRowSum ? D + 16 : D;  // MMA N of the P.V product
  static constexpr int kOnesBytes = kTensorRowSum ? BN * 128 : 0;  // 128 keys x 64 columns of fp16 1.0
  static constexpr int kSmemBytes =
      kQBytes + kStages * kTileBytes + kStageBufs * kStageBytes + kOnesBytes + 1024;  // + alignment slack
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

struct Params {
  __nv_bfloat16* o;
  float* lse;
  int Hq, Hkv, G, Sq, Sk;
  int causal;     // 0 none, else key j allowed for row i iff j <= i + diag
  int diag;
  int n_qblocks;  // ceil(Sq / ROWS_PER_ITEM)
  int BH;         // B * Hq
  int n_items;    // BH * n_qblocks (* n_splits)
  float c;        // scale * log2(e)
  // split-key mode: the key tiles of each (b, h, query block) are cut into n_splits
  // contiguous ranges; each writes an fp32 partial O and LSE for the merge
  int n_splits;
  float* o_part;    // [n_splits][BH][Sq][D]
  float* lse_part;  // [n_splits][BH][Sq]
  int sched_slot;   // which schedule counter this launch claims items from
  // block-sparse mode: bit-packed mask [B][mask_heads][n_qtiles][mask_words], one bit per
  // (128-row query block, 128-key block), bit kb % 32 of word kb / 32
  const uint32_t* mask;
  int mask_heads;  // 1 (one mask for every head) or Hq
  int mask_words;  // words per mask row: ceil(ceil(Sk / 128) / 32)
  int n_qtiles;    // ceil(Sq / 128)
  // ordered mode: key-tile order [B][order_heads][n_qblocks][order_len], one row per
  // 256-row query block (the item), visited in row order
  const int32_t* order;
  int order_heads;  // 1 (one order for every head) or Hq
  int order_len;    // entries per row: ceil(Sk / 128)
};

struct Item {
  int bh;       // b * Hq + query head
  int kv_z;     // b * Hkv + kv head
  int q0;       // first query row
  int j0;       // first key tile
  int n_tiles;  // key tiles to visit
  int split;    // key range index (split-key mode)
};

// Item x of the heaviest-first list: query block from the last, then (split-key
// mode) the key range, heads fastest.  Grouped order (GROUPED; dense, block-sparse
// and ordered modes): the G x n_qblocks items that read one kv head's K and V are
// adjacent -- kv heads in order, then query blocks from the last, the group's
// query heads fastest -- so they run side by side and share each K and V tile
// through L2.
template <bool SPLIT, bool SPARSE = false, bool GROUPED = false>
__device__ __forceinline__ Item item_at(const Params& p, int x) {
  Item it;
  int qb, r;
  if constexpr (GROUPED) {
    const int per = p.G * p.n_qblocks;  // items of one kv head
    const int grp = x / per, w = x % per;
    qb = p.n_qblocks - 1 - w / p.G;
    it.bh = (grp / p.Hkv) * p.Hq + (grp % p.Hkv) * p.G + w % p.G;
    it.split = 0;
  } else if (SPLIT) {
    const int per = p.BH * p.n_splits;
    qb = p.n_qblocks - 1 - x / per;
    r = x % per;
    it.split = r / p.BH;
    it.bh = r % p.BH;
  } else {
    qb = p.n_qblocks - 1 - x / p.BH;
    it.bh = x % p.BH;
    it.split = 0;
  }
  const int b = it.bh / p.Hq;
  const int hq = it.bh % p.Hq;
  it.kv_z = b * p.Hkv + hq / p.G;
  it.q0 = qb * ROWS_PER_ITEM;
  int kv_end = p.Sk;
  if (p.causal) {
    const int last_row = min(it.q0 + ROWS_PER_ITEM, p.Sq) - 1;
    kv_end = min(p.Sk, last_row + p.diag + 1);
  }
  const int n_full = kv_end > 0 ? (kv_end + BN - 1) / BN : 0;
  if (SPLIT) {
    it.j0 = static_cast<int>(static_cast<int64_t>(it.split) * n_full / p.n_splits);
    it.n_tiles = static_cast<int>(static_cast<int64_t>(it.split + 1) * n_full / p.n_splits) - it.j0;
  } else {
    it.j0 = 0;
    it.n_tiles = n_full;  // block-sparse mode: the causal bound; the producer counts the marked tiles
  }
  return it;
}

// Block-sparse mode: the two mask rows of an item (its Q tiles' query blocks; a Q
// tile past the last query block has none), word w of their union clipped to the
// item's causal key-tile bound n_full, and that tile's own bits.
struct MaskRows {
  const uint32_t* r0;  // Q tile 0's row
  const uint32_t* r1;  // Q tile 1's row, or nullptr
};

__device__ __forceinline__ MaskRows mask_rows(const Params& p, const Item& it) {
  const int b = it.bh / p.Hq;
  const int hm = p.mask_heads == 1 ? 0 : it.bh % p.Hq;
  const int qt = it.q0 / BM;
  const uint32_t* base = p.mask + (static_cast<int64_t>(b) * p.mask_heads + hm) * p.n_qtiles * p.mask_words;
  MaskRows m;
  m.r0 = base + static_cast<int64_t>(qt) * p.mask_words;
  m.r1 = qt + 1 < p.n_qtiles ? m.r0 + p.mask_words : nullptr;
  return m;
}

// bits of word w kept by a key-tile bound n (tiles 0 .. n-1)
__device__ __forceinline__ uint32_t bound_bits(int w, int n) {
  const int left = n - 32 * w;
  return left >= 32 ? 0xFFFFFFFFu : (left <= 0 ? 0u : ((1u << left) - 1u));
}

__device__ __forceinline__ uint32_t union_word(const MaskRows& m, int w, int n) {
  const uint32_t u = __ldg(m.r0 + w) | (m.r1 ? __ldg(m.r1 + w) : 0u);
  return u & bound_bits(w, n);
}

// number of key tiles the item visits: the marked tiles within its causal bound (the
// lanes of the calling warp take one word each)
__device__ __forceinline__ int sparse_tiles(const Params& p, const Item& it) {
  const MaskRows m = mask_rows(p, it);
  const int lane = static_cast<int>(threadIdx.x % 32);
  int n = 0;
  for (int w0 = 0; w0 * 32 < it.n_tiles; w0 += 32) {
    const int w = w0 + lane;
    int c = w * 32 < it.n_tiles ? __popc(union_word(m, w, it.n_tiles)) : 0;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) c += __shfl_xor_sync(0xffffffffu, c, off);
    n += c;
  }
  return n;
}

// Ordered mode (the priority-ordered visitation of page "CoSA: Accelerating Long-Context
// Inference via Proxy-Kernel Co-Designed Sparse Attention": the kernel reads the key
// tiles in the order a priority list gives).  An item visits, in row order, every
// entry e of its row with 0 <= e < its causal key-tile bound.  The row is scanned 32
// entries at a time: each lane holds one entry of the current window and a ballot
// marks the entries visited, so a warp finds the next tile with find-first-set and a
// shuffle instead of a chain of dependent loads.
__device__ __forceinline__ const int32_t* order_row(const Params& p, const Item& it) {
  const int b = it.bh / p.Hq;
  const int ho = p.order_heads == 1 ? 0 : it.bh % p.Hq;
  const int qb = it.q0 / ROWS_PER_ITEM;
  return p.order + ((static_cast<int64_t>(b) * p.order_heads + ho) * p.n_qblocks + qb) * p.order_len;
}

// window w of an order row: this lane's entry in `val` (-1 past the row), and the
// ballot of the entries visited under the key-tile bound n
__device__ __forceinline__ uint32_t order_window(const int32_t* row, int len, int w, int n, int& val) {
  const int e = 32 * w + static_cast<int>(threadIdx.x % 32);
  val = e < len ? __ldg(row + e) : -1;
  return __ballot_sync(0xffffffffu, val >= 0 && val < n);
}

// number of key tiles an item visits in ordered mode (the whole warp calls it; four
// windows' loads are in flight together)
__device__ __forceinline__ int ordered_tiles(const Params& p, const Item& it) {
  const int32_t* row = order_row(p, it);
  const int lane = static_cast<int>(threadIdx.x % 32);
  int n = 0;
  for (int w0 = 0; 32 * w0 < p.order_len; w0 += 4) {
    int v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int e = 32 * (w0 + u) + lane;
      v[u] = e < p.order_len ? __ldg(row + e) : -1;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) n += __popc(__ballot_sync(0xffffffffu, v[u] >= 0 && v[u] < it.n_tiles));
  }
  return n;
}

// Walks the visited entries of an order row, one window at a time (warp-uniform).
struct OrderWalk {
  const int32_t* row = nullptr;
  int len = 0, bound = 0, w = 0, val = -1;
  uint32_t cur = 0;
  __device__ __forceinline__ void start(const int32_t* r, int l, int n) {
    row = r;
    len = l;
    bound = n;
    w = 0;
    cur = order_window(row, len, 0, bound, val);
  }
  // the next visited tile (0 if the row has no more, which the counts rule out
  // unless the row changed under the call)
  __device__ __forceinline__ int next() {
    const int w_end = (len + 31) / 32;
    while (cur == 0 && w + 1 < w_end) cur = order_window(row, len, ++w, bound, val);
    const int bit = cur ? __ffs(cur) - 1 : 0;
    const int tile = __shfl_sync(0xffffffffu, val, bit);
    const bool found = cur != 0;
    cur &= cur - 1;
    return found ? tile : 0;
  }
};

__device__ int g_status;  // sticky: 0 = fine, else the site of the first wait that ran out

#ifdef ATTN_TRACE
// Timeline build (-DATTN_TRACE, off by default): lane 0 of each role records
// (%globaltimer, event, argument) at the points below, in a fixed device array
// that attn_fwd_trace_read copies out.  Event codes and roles are listed in
// attn_fwd_trace.h.  Without the switch every trace point compiles to nothing.
constexpr int kTraceRoles = 5;      // producer, issuer, softmax tile 0, softmax tile 1, store warp
constexpr int kTraceEvents = 2048;  // per role and CTA; later events are counted but not kept
constexpr int kTraceCtas = 160;     // CTAs numbered past this are not recorded
struct TraceRec {
  unsigned long long t;
  unsigned int code;
  unsigned int arg;
};
__device__ TraceRec g_trace[kTraceCtas * kTraceRoles * kTraceEvents];
__device__ unsigned int g_trace_n[kTraceCtas * kTraceRoles];
struct Tracer {
  int role;
  bool on;  // the recording lane
  unsigned int n;
  __device__ __forceinline__ void rec(unsigned int code, unsigned int arg) {
    if (!on) return;
    if (blockIdx.x < kTraceCtas && n < kTraceEvents)
      g_trace[(blockIdx.x * kTraceRoles + role) * kTraceEvents + n] = TraceRec{global_timer_ns(), code, arg};
    ++n;
  }
  __device__ __forceinline__ void done() {
    if (on && blockIdx.x < kTraceCtas) g_trace_n[blockIdx.x * kTraceRoles + role] = n;
  }
};
#define ATTN_TR_DECL(role, on) Tracer tr_{(role), (on), 0u}
#define ATTN_TR(code, arg) tr_.rec((code), static_cast<unsigned int>(arg))
#define ATTN_TR_DONE() tr_.done()
#else
#define ATTN_TR_DECL(role, on) ((void)0)
#define ATTN_TR(code, arg) ((void)0)
#define ATTN_TR_DONE() ((void)0)
#endif

// Dynamic schedule.  CTA c starts on item c; later items are claimed in list
// order (heaviest first) from a counter, so a CTA that finishes early takes the
// next item and the CTAs end within about one (small) item of each other.  Each
// launch uses one of kSchedSlots counters, chosen by the host: launches made
// directly take the first kEagerSlots in turn, launches recorded into a CUDA graph
// (stream capture) the remaining ones in turn, so a graph's launches, which keep
// the counter they were recorded with, never share one with a direct launch.  Every CTA
// claims until a claim comes back past the last item, so a launch makes exactly
// n_items claims (a CTA that unwinds early makes the rest of its claims before it
// exits); the claim numbered n_items - 1 is the launch's last, and its taker
// returns the counter to zero, with no end-of-kernel synchronisation.
constexpr int kEagerSlots = 64;
constexpr int kCaptureSlots = 4096;
constexpr int kSchedSlots = kEagerSlots + kCaptureSlots;
__device__ int g_sched_next[kSchedSlots];
constexpr int kSeqSlots = 4;  // depth of the shared-memory ring through which the producer publishes items
constexpr int kSeqConsumers = 10;  // warps reading the ring: eight softmax warps, the issuer, the store warp

__device__ __forceinline__ uint8_t* align_1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~static_cast<uintptr_t>(1023));
}

// Every lane polls; the answer is made warp-uniform so the .sync.aligned
// tcgen05 instructions that follow are always executed by the whole warp.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile uint32_t* abort_flag,
                                          uint64_t timeout_ns) {
  const bool ok = mbar_wait_bounded(bar, parity, abort_flag, timeout_ns);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void record_abort(volatile uint32_t* abort_flag, int site) {
  *abort_flag = 1;
  atomicCAS(&g_status, 0, site);
}

template <int D, bool SPLIT, bool SPARSE, bool ORDERED = false, bool GROUPED = false>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap to,
                    const Params p) {
  using C = Cfg<D>;
  constexpr int S = C::kStages;
  // block-sparse and ordered modes: the producer counts each item's key tiles and
  // publishes the count with the item; every role walks the same tile sequence
  constexpr bool LISTED = SPARSE || ORDERED;
  static_assert(!(SPARSE && ORDERED) && !(SPLIT && (SPARSE || ORDERED)), "one visiting mode at a time");
  static_assert(!GROUPED || !SPLIT, "the grouped order lists whole-key-range items");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_1024(smem_raw);
  uint8_t* q_s = smem;               // Q tile t at q_s + t * kTileBytes
  uint8_t* kv_s = smem + C::kQBytes;  // slot s at kv_s + s * kTileBytes
  uint8_t* st_s = kv_s + S * C::kTileBytes;  // O staging buffer b at st_s + b * kStageBytes
  uint8_t* ones_s = st_s + C::kStageBufs * C::kStageBytes;  // D = 64: the ones block of the row-sum columns
  __shared__ uint64_t kv_full[S], kv_empty[S];
  __shared__ uint64_t v_ready[S];  // a V tile in slot s has been converted to fp16 (odd slots only)
  __shared__ uint64_t q_full, q_empty, s_full[QTILES], p_full[QTILES], o_final[QTILES], o_empty[QTILES];
  __shared__ uint64_t stage_full[QTILES], stage_rel[QTILES], mma_drain;
  __shared__ uint64_t seq_full[kSeqSlots], seq_empty[kSeqSlots];
  __shared__ int item_seq[kSeqSlots];  // the CTA's k-th item at slot k % kSeqSlots (-1: no more)
  __shared__ int item_ntiles[kSeqSlots];  // block-sparse / ordered mode: its key tiles (counted by the producer)
  __shared__ uint32_t tmem_base_slot;
  __shared__ uint32_t abort_flag;

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
      mbar_init(&v_ready[s], 8);  // one arrival per softmax warp
    }
    mbar_init(&q_full, 1);
    mbar_init(&q_empty, 1);
    for (int t = 0; t < QTILES; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], 4 * 32);
      mbar_init(&o_empty[t], 4 * 32);
      mbar_init(&o_final[t], 1);
      mbar_init(&stage_full[t], 4 * 32);
      mbar_init(&stage_rel[t], 1);
    }
    mbar_init(&mma_drain, 1);
    for (int i = 0; i < kSeqSlots; ++i) {
      mbar_init(&seq_full[i], 1);
      mbar_init(&seq_empty[i], kSeqConsumers);
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&tmem_base_slot, kTmemCols);
    tmem_relinquish();
  }
  if constexpr (C::kTensorRowSum) {
    // fp16 1.0 everywhere (the swizzle does not matter for a constant block), made
    // visible to the tensor cores' (async proxy) reads
    for (int i = threadIdx.x; i < C::kOnesBytes / 16; i += kThreads)
      reinterpret_cast<uint4*>(ones_s)[i] = make_uint4(0x3C003C00u, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u);
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_slot;
  volatile uint32_t* abort_v = &abort_flag;
  // k-th item of this CTA as published by the producer (-1: no more); false when a wait gave up
  auto next_item = [&](int k, int& x, int* ntiles = nullptr) {
    if (!warp_wait(&seq_full[k % kSeqSlots], (k / kSeqSlots) & 1, abort_v, kTimeoutNs)) return false;
    x = *reinterpret_cast<volatile int*>(&item_seq[k % kSeqSlots]);
    if (ntiles) *ntiles = *reinterpret_cast<volatile int*>(&item_ntiles[k % kSeqSlots]);
    __syncwarp();
    if (lane == 0) mbar_arrive(&seq_empty[k % kSeqSlots]);
    return true;
  };

  if (warp >= 8) {
   // warpgroup 2: every warp shrinks its registers at the same instruction, then splits by role
   regs_decrease<kRegsOther>();
   if (warp == kLoadWarp) {
    // ------------------------------------------------------------ TMA producer
    ATTN_TR_DECL(0, lane == 0);
    ATTN_TR(0, 0);  // CTA start
    if (lane == 0) {
      tma_prefetch_map(&tq);
      tma_prefetch_map(&tk);
      tma_prefetch_map(&tv);
    }
    uint32_t kv_it = 0;     // K/V loads issued so far (over all items)
    uint32_t q_issued = 0;  // Q loads issued so far (one per item with key tiles)
    bool ok = true;
    int x = static_cast<int>(blockIdx.x);  // the first item is fixed; the rest are claimed
    for (int k = 0; ok; ++k) {
      const bool more = x < p.n_items;
      // publish the item to the other roles
      if (k >= kSeqSlots) {
        ok = warp_wait(&seq_empty[k % kSeqSlots], (k / kSeqSlots - 1) & 1, abort_v, kTimeoutNs);
        if (!ok) break;
      }
      int n_marked = 0;  // block-sparse / ordered mode: the key tiles the item visits
      if constexpr (SPARSE) {
        if (more) n_marked = sparse_tiles(p, item_at<SPLIT, SPARSE, GROUPED>(p, x));
      } else if constexpr (ORDERED) {
        if (more) n_marked = ordered_tiles(p, item_at<SPLIT, false, GROUPED>(p, x));
      }
      if (lane == 0) {
        item_seq[k % kSeqSlots] = more ? x : -1;
        if constexpr (LISTED) item_ntiles[k % kSeqSlots] = n_marked;
        mbar_arrive(&seq_full[k % kSeqSlots]);
      }
      __syncwarp();
      ATTN_TR(1, more ? x : -1);  // item published
      if (!more) break;
      const Item it = item_at<SPLIT, SPARSE, GROUPED>(p, x);
      const int n_tiles = LISTED ? n_marked : it.n_tiles;
      // The next item is claimed once this item's loads are all issued (about two
      // key tiles before its end), so items are handed out in the order CTAs free up.
      auto claim = [&]() {
        int claimed = 0;
        if (lane == 0) {
          claimed = atomicAdd(&g_sched_next[p.sched_slot], 1);
          if (claimed == p.n_items - 1) g_sched_next[p.sched_slot] = 0;  // the launch's last claim
        }
        return static_cast<int>(gridDim.x) + __shfl_sync(0xffffffffu, claimed, 0);
      };
      if (n_tiles == 0) {
        x = claim();
        continue;
      }
      if (q_issued > 0) {  // the previous item's last S has finished reading Q
        ok = warp_wait(&q_empty, (q_issued - 1) & 1, abort_v, kTimeoutNs);
        if (!ok) break;
      }
      mbar_arrive_expect_tx_elect(&q_full, C::kQBytes);
#pragma unroll
      for (int t = 0; t < QTILES; ++t)
#pragma unroll
        for (int cb = 0; cb < D / 64; ++cb)
          tma_load_3d_elect(q_s + t * C::kTileBytes + cb * C::kColBlockBytes, &tq, &q_full, cb * 64, it.q0 + t * BM,
                            it.bh);
      ++q_issued;
      // block-sparse mode: the marked key tiles in order (find-first-set over the union words)
      MaskRows mrows{};
      int mw = 0;
      uint32_t mcur = 0;
      int kb = 0;
      if constexpr (SPARSE) {
        mrows = mask_rows(p, it);
        mcur = union_word(mrows, 0, it.n_tiles);
      }
      OrderWalk owalk;  // ordered mode: the item's row of the order
      if constexpr (ORDERED) owalk.start(order_row(p, it), p.order_len, it.n_tiles);
      for (int i = 0; i < 2 * n_tiles; ++i) {  // K_j is load 2j, V_j is load 2j+1
        const uint32_t slot = kv_it % S;
        const uint32_t use = kv_it / S;
        if (use > 0) {
          ok = warp_wait(&kv_empty[slot], (use - 1) & 1, abort_v, kTimeoutNs);
          if (!ok) break;
        }
        const CUtensorMap* map = (i & 1) ? &tv : &tk;
        if constexpr (SPARSE) {
          if (!(i & 1)) {  // the next marked tile (the item has n_tiles of them)
            const int mw_end = (it.n_tiles + 31) / 32;  // bounded even if the mask changed under the call
            while (mcur == 0 && mw + 1 < mw_end) mcur = union_word(mrows, ++mw, it.n_tiles);
            kb = mcur ? 32 * mw + __ffs(mcur) - 1 : 0;
            mcur &= mcur - 1;
          }
        } else if constexpr (ORDERED) {
          if (!(i & 1)) kb = owalk.next();  // the next tile of the order
        } else {
          kb = it.j0 + (i >> 1);
        }
        mbar_arrive_expect_tx_elect(&kv_full[slot], C::kTileBytes);
#pragma unroll
        for (int cb = 0; cb < D / 64; ++cb)
          tma_load_3d_elect(kv_s + slot * C::kTileBytes + cb * C::kColBlockBytes, map, &kv_full[slot], cb * 64,
                            kb * BN, it.kv_z);
        ATTN_TR((i & 1) ? 3 : 2, kb);  // V or K load issued
        ++kv_it;
      }
      if (ok) x = claim();
    }
    if (!ok) {
      if (lane == 0) {
        record_abort(abort_v, kSiteProducer);
        // the claims this CTA has not made yet, up to its first one past the last item,
        // so the launch still makes n_items claims and its last taker resets the counter
        while (x < p.n_items) {
          const int claimed = atomicAdd(&g_sched_next[p.sched_slot], 1);
          if (claimed == p.n_items - 1) g_sched_next[p.sched_slot] = 0;
          x = static_cast<int>(gridDim.x) + claimed;
        }
      }
      // unwinding: let the copies already in flight land before the CTA exits
      if (q_issued > 0) mbar_wait_bounded(&q_full, (q_issued - 1) & 1, abort_v, kDrainTimeoutNs);
      for (uint32_t i = (kv_it > S ? kv_it - S : 0); i < kv_it; ++i)
        mbar_wait_bounded(&kv_full[i % S], (i / S) & 1, abort_v, kDrainTimeoutNs);
    }
    ATTN_TR_DONE();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ tcgen05 issuer
    const uint32_t idesc_s = idesc_bf16_f32(BM, BN, false);
    const uint32_t idesc_pv = idesc_f16_f32(BM, C::kPvN, true);  // fp16 P (TMEM) times fp16 V (smem)
    const uint32_t q_addr = smem_u32(q_s);
    const uint32_t kv_addr = smem_u32(kv_s);
    // The whole warp runs the issue code (converged); one elected lane issues.
    // Operand descriptors are built once per tile; a K step moves the start
    // address field (bits 0-13, address >> 4) by a constant, never carrying out.
    // each issue ends with commits to up to two mbarriers (kNoBar: none)
    auto issue_s = [=](int t, uint32_t slot, uint32_t bar0 = kNoBar, uint32_t bar1 = kNoBar) {
      const uint64_t qd = sdesc_sw128(opaque(q_addr) + t * C::kTileBytes, 16, 1024);
      const uint64_t kd = sdesc_sw128(kv_addr + slot * C::kTileBytes, 16, 1024);
      static_assert(C::kColBlockBytes == 16384, "K-step offsets of mma_bf16_ss_k8");
      if constexpr (D == 128)
        mma_bf16_ss_k8(tmem + t * BN, qd, kd, idesc_s, bar0, bar1);
      else
        mma_bf16_ss_k4(tmem + t * BN, qd, kd, idesc_s, bar0, bar1);
    };
    const uint32_t ones_addr = smem_u32(ones_s);
    auto issue_pv = [=](int t, uint32_t slot, bool accumulate, uint32_t bar0 = kNoBar, uint32_t bar1 = kNoBar) {
      // V is MN-major: the leading byte offset steps from one 64-column block of V to
      // the next; at D = 64 the second block is the ones block (the row-sum columns)
      const uint32_t v_addr = opaque(kv_addr) + slot * C::kTileBytes;
      const uint64_t vd =
          sdesc_sw128(v_addr, C::kTensorRowSum ? ones_addr - v_addr : C::kColBlockBytes, 1024);
      static_assert(BN == 128, "K steps of mma_bf16_ts_k8");
      mma_bf16_ts_k8(tmem + 2 * BN + t * 128, tmem + t * BN + 64, vd, idesc_pv, accumulate ? 1u : 0u, bar0, bar1);
    };
    // wait for load number `n` of the K/V stream (a K tile), or for its conversion (a V tile)
    auto wait_kv = [&](uint32_t n) {
      return warp_wait(&kv_full[n % S], (n / S) & 1, abort_v, kTimeoutNs);
    };
    auto wait_v = [&](uint32_t n) {
      return warp_wait(&v_ready[n % S], (n / S) & 1, abort_v, kTimeoutNs);
    };
    ATTN_TR_DECL(1, lane == 0);
    uint32_t kv_it = 0;   // K/V loads consumed
    uint32_t g = 0;       // key tiles processed over all items (p_full phase)
    uint32_t n_done = 0;  // items with key tiles processed
    bool ok = true;
    for (int k = 0; ok; ++k) {
      int x, n_marked = 0;
      ok = next_item(k, x, LISTED ? &n_marked : nullptr);
      if (!ok || x < 0) break;
      const int n = LISTED ? n_marked : item_at<SPLIT, false, GROUPED>(p, x).n_tiles;
      if (n == 0) continue;
      ok = warp_wait(&q_full, n_done & 1, abort_v, kTimeoutNs);
      if (ok) ok = wait_kv(kv_it);
      if (!ok) break;
      uint32_t kslot = kv_it % S;
      ++kv_it;
      tc_fence_after();
      ATTN_TR(12, x);  // item start: its first S products
      issue_s(0, kslot, smem_u32(&s_full[0]));
      issue_s(1, kslot, smem_u32(&s_full[1]), smem_u32(&kv_empty[kslot]));
      if (n == 1) mma_commit_elect(&q_empty);
      // One step: P.V of both Q tiles on V_j and, unless it is the item's last, their S on K_(j+1).
      // At D = 64, where the softmax sets the pace, the first, second-last and last steps are separate
      // compile-time variants, so the steady-state step carries no per-step test; with the K wait below moved
      // ahead of the hand-off, 3.5 % faster on a chunked prefill at D = 64 (no gain at D = 128, which keeps the
      // plain loop).
      auto step = [&](auto first_c, auto last_c, auto qlast_c) -> bool {
        constexpr bool first = decltype(first_c)::value;  // j == 0: the O_t of the previous item must be read out
        constexpr bool last = decltype(last_c)::value;    // j == n - 1: the P.V complete O_t
        constexpr bool qlast = decltype(qlast_c)::value;  // j == n - 2: the S issued here are the item's last
        const uint32_t vslot = kv_it % S;
        bool good = wait_v(kv_it);
        ++kv_it;
        // K_(j+1) is awaited here, before the softmax hand-off, not between P.V_0 and S_0 (its ring slot
        // was released steps ago, so the wait does not depend on this step's products)
        uint32_t ks = 0;
        if constexpr (!last) {
          ks = kv_it % S;
          if (good) good = wait_kv(kv_it);
          ++kv_it;
        }
        if constexpr (first) {
          if (good && n_done > 0) good = warp_wait(&o_empty[0], (n_done - 1) & 1, abort_v, kTimeoutNs);
        }
        if (good) good = warp_wait(&p_full[0], g & 1, abort_v, kTimeoutNs);
        if (!good) return false;
        tc_fence_after();
        // the last P.V of O_0 completes it: its epilogue can start
        issue_pv(0, vslot, !first, last ? smem_u32(&o_final[0]) : kNoBar);
        ATTN_TR(11, 0);
        if constexpr (!last) issue_s(0, ks, smem_u32(&s_full[0]));
        if constexpr (first) {
          if (n_done > 0) good = warp_wait(&o_empty[1], (n_done - 1) & 1, abort_v, kTimeoutNs);
        }
        if (good) good = warp_wait(&p_full[1], g & 1, abort_v, kTimeoutNs);
        if (!good) return false;
        tc_fence_after();
        issue_pv(1, vslot, !first, last ? smem_u32(&o_final[1]) : kNoBar, smem_u32(&kv_empty[vslot]));
        ATTN_TR(11, 1);
        if constexpr (!last) {
          issue_s(1, ks, smem_u32(&s_full[1]), smem_u32(&kv_empty[ks]));
          if constexpr (qlast) mma_commit_elect(&q_empty);  // that was the item's last S
        }
        ++g;
        return true;
      };
      if constexpr (D == 64) {
        using T = std::true_type;
        using F = std::false_type;
        if (n == 1) {
          ok = step(T{}, T{}, F{});
        } else {
          ok = (n == 2) ? step(T{}, F{}, T{}) : step(T{}, F{}, F{});
          for (int j = 1; ok && j + 2 < n; ++j) ok = step(F{}, F{}, F{});
          if (ok && n >= 3) ok = step(F{}, F{}, T{});
          if (ok) ok = step(F{}, T{}, F{});
        }
      } else {
        for (int j = 0; j < n; ++j) {
          const uint32_t vslot = kv_it % S;
          ok = wait_v(kv_it);
          ++kv_it;
          if (ok && j == 0 && n_done > 0) ok = warp_wait(&o_empty[0], (n_done - 1) & 1, abort_v, kTimeoutNs);
          if (ok) ok = warp_wait(&p_full[0], g & 1, abort_v, kTimeoutNs);
          if (!ok) break;
          tc_fence_after();
          // the last P.V of O_0 completes it: its epilogue can start
          issue_pv(0, vslot, j > 0, j + 1 == n ? smem_u32(&o_final[0]) : kNoBar);
          ATTN_TR(11, 0);  // P.V of Q tile 0 issued
          const bool more = j + 1 < n;
          if (more) {
            kslot = kv_it % S;
            ok = wait_kv(kv_it);
            ++kv_it;
            if (!ok) break;
            tc_fence_after();
            issue_s(0, kslot, smem_u32(&s_full[0]));
          }
          if (j == 0 && n_done > 0) ok = warp_wait(&o_empty[1], (n_done - 1) & 1, abort_v, kTimeoutNs);
          if (ok) ok = warp_wait(&p_full[1], g & 1, abort_v, kTimeoutNs);
          if (!ok) break;
          tc_fence_after();
          issue_pv(1, vslot, j > 0, j + 1 == n ? smem_u32(&o_final[1]) : kNoBar, smem_u32(&kv_empty[vslot]));
          ATTN_TR(11, 1);  // P.V of Q tile 1 issued
          if (more) {
            issue_s(1, kslot, smem_u32(&s_full[1]), smem_u32(&kv_empty[kslot]));
            if (j + 2 == n) mma_commit_elect(&q_empty);  // that was the item's last S
          }
          ++g;
        }
      }
      if (!ok) break;
      ++n_done;
    }
    if (!ok && lane == 0) record_abort(abort_v, kSiteIssuer);
    // every MMA issued above has completed before TMEM can be freed
    mma_commit_elect(&mma_drain);
    warp_wait(&mma_drain, 0, abort_v, ok ? kTimeoutNs : kDrainTimeoutNs);
    ATTN_TR(13, 0);  // every MMA of the CTA has completed
    ATTN_TR_DONE();
   } else if (warp == kStoreWarp) {
    // ------------------------------------------------------------ O stores
    // Once a Q tile's epilogue has staged O (stage_full), one TMA store per 64
    // columns writes it out; the staging buffer is handed back (stage_rel) when the
    // stores have read it.  The softmax warps never wait for a store.
    uint32_t e_seen[QTILES] = {0, 0};
    ATTN_TR_DECL(4, lane == 0);
    bool ok = true;
    for (int k = 0; ok; ++k) {
      int x, n_marked = 0;
      ok = next_item(k, x, LISTED ? &n_marked : nullptr);
      if (!ok || x < 0) break;
      if constexpr (!SPLIT) {  // split-key partials are written by the softmax warps directly
        const Item it = item_at<SPLIT, SPARSE, GROUPED>(p, x);
        if ((LISTED ? n_marked : it.n_tiles) == 0) continue;
        for (int t = 0; t < QTILES && ok; ++t) {
          ok = warp_wait(&stage_full[t], e_seen[t] & 1, abort_v, kTimeoutNs);
          if (!ok) break;
          ++e_seen[t];
          uint8_t* stage = st_s + ((C::kStageBufs == 1) ? 0 : t) * C::kStageBytes;
#pragma unroll
          for (int cb = 0; cb < D / 64; ++cb)
            tma_store_3d_elect(&to, stage + cb * (BM * 128), cb * 64, it.q0 + t * BM, it.bh);
          bulk_commit_group_elect();
          ATTN_TR(30, t);  // O stores of Q tile t issued
          bulk_wait_group_read0();  // the staging tile has been read: hand it on
          __syncwarp();
          if (lane == 0) mbar_arrive(&stage_rel[t]);
        }
      }
    }
    if (!ok && lane == 0) record_abort(abort_v, kSiteEpilogue);
    bulk_wait_group0();  // every store has landed before the CTA exits
    ATTN_TR(31, 0);
    ATTN_TR_DONE();
   }
  } else {
    // ------------------------------------------------------------ softmax (+ rescale, epilogue)
    regs_increase<kRegsSoftmax>();
    const int t = warp / 4;
    const int quarter = warp % 4;
    ATTN_TR_DECL(2 + t, quarter == 0 && lane == 0);
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t s_tmem = tmem + lane_off + t * BN;
    const uint32_t o_tmem = tmem + lane_off + 2 * BN + t * 128;
    const float c = p.c;
    uint32_t g = 0;       // key tiles processed over all items (s_full phase)
    uint32_t n_done = 0;  // items with key tiles processed (o_final[t] and staging phase)
    bool ok = true;

    for (int k = 0; ok; ++k) {
      int x, n_marked = 0;
      ok = next_item(k, x, LISTED ? &n_marked : nullptr);
      if (!ok) {
        if (lane == 0) record_abort(abort_v, kSiteSoftmax);
        break;
      }
      if (x < 0) break;
      const Item it = item_at<SPLIT, SPARSE, GROUPED>(p, x);
      const int n_tiles = LISTED ? n_marked : it.n_tiles;  // key tiles the item visits
      const int row = it.q0 + t * BM + quarter * 32 + lane;  // global query row
      const bool live = row < p.Sq;
      __nv_bfloat16* orow = p.o + (static_cast<int64_t>(it.bh) * p.Sq + row) * D;
      float* lrow = p.lse + static_cast<int64_t>(it.bh) * p.Sq + row;
      // split-key mode: this item's partial result rows
      const int64_t prow = (static_cast<int64_t>(it.split) * p.BH + it.bh) * p.Sq + row;
      if (n_tiles == 0) {  // no key is visible to any row of this item (or its key range is empty)
        if (live) {
          if (SPLIT) {
            float4* dst = reinterpret_cast<float4*>(p.o_part + prow * D);
#pragma unroll
            for (int v4 = 0; v4 < D / 4; ++v4) dst[v4] = make_float4(0.f, 0.f, 0.f, 0.f);
            p.lse_part[prow] = -INFINITY;
          } else {
            uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
            for (int v4 = 0; v4 < D / 8; ++v4) dst[v4] = make_uint4(0u, 0u, 0u, 0u);
            *lrow = -INFINITY;
          }
        }
        continue;
      }
      // last allowed key of this row, and of the tile's first row (the most restricted)
      const int tile_row0 = it.q0 + t * BM;
      int lim = p.Sk - 1, lim_tile = p.Sk - 1;
      if (p.causal) {
        lim = min(lim, row + p.diag);
        lim_tile = min(lim_tile, tile_row0 + p.diag);
      }
      float m = -INFINITY;   // running max, log2 units
      float l = 0.0f;        // sum of the fp16-rounded P the tensor cores use (normalises O)
      float l_exact = 0.0f;  // sum of the fp32 P (gives LSE)

      // block-sparse mode: walk the same marked tiles as the producer; a tile that only
      // the other Q tile's query block marks is wholly masked for this one
      MaskRows mrows{};
      int mw = 0;
      uint32_t mcur = 0, mown = 0;
      if constexpr (SPARSE) {
        mrows = mask_rows(p, it);
        mcur = union_word(mrows, 0, it.n_tiles);
        mown = t == 0 ? __ldg(mrows.r0) : (mrows.r1 ? __ldg(mrows.r1) : 0u);
      }
      OrderWalk owalk;  // ordered mode: the same walk as the producer's
      if constexpr (ORDERED) owalk.start(order_row(p, it), p.order_len, it.n_tiles);
      for (int j = 0; j < n_tiles; ++j, ++g) {
        // the tile's index first (its loads overlap the wait for S)
        int jg = it.j0 + j;  // key tile index within the head
        bool own = true;     // block-sparse mode: this Q tile's query block marks the tile
        if constexpr (SPARSE) {
          const int mw_end = (it.n_tiles + 31) / 32;
          while (mcur == 0 && mw + 1 < mw_end) {
            mcur = union_word(mrows, ++mw, it.n_tiles);
            mown = t == 0 ? __ldg(mrows.r0 + mw) : (mrows.r1 ? __ldg(mrows.r1 + mw) : 0u);
          }
          const int bit = mcur ? __ffs(mcur) - 1 : 0;
          jg = 32 * mw + bit;
          own = (mown >> bit) & 1u;
          mcur &= mcur - 1;
        } else if constexpr (ORDERED) {
          jg = owalk.next();
        }
        // the tile is unmarked for this Q tile, or straddles the diagonal or the end of K
        const bool masked = !own || jg * BN + BN - 1 > lim_tile;
        const int kmax = own ? lim - jg * BN : -1;
        // V of this tile (load 2g + 1 of the CTA's K/V stream) to fp16, in place in its ring
        // slot: the 256 softmax threads take one 16-byte chunk in 256 each (a chunk holds 8
        // consecutive values of one row, so the swizzled layout is unchanged), make their
        // writes visible to the tensor cores and arrive on v_ready.  This runs between the
        // previous tile's hand-off and the wait for this tile's S, while the tensor cores
        // work on the P.V and S products issued in between; the slot is refilled only after
        // the P.V that waited for v_ready has read it.
        {
          const uint32_t vn = 2u * g + 1u;
          ok = warp_wait(&kv_full[vn % S], (vn / S) & 1, abort_v, kTimeoutNs);
          if (!ok) break;
          constexpr int kChunks = C::kTileBytes / 16 / 256;  // per thread: 8 (D = 128) or 4 (D = 64)
          const uint32_t base = smem_u32(kv_s + (vn % S) * C::kTileBytes) + 16u * threadIdx.x;
          uint4 w[kChunks];
#pragma unroll
          for (int u = 0; u < kChunks; ++u) w[u] = lds128(base + 4096u * u);
#pragma unroll
          for (int u = 0; u < kChunks; ++u) {
            w[u].x = bf16x2_to_f16x2(w[u].x);
            w[u].y = bf16x2_to_f16x2(w[u].y);
            w[u].z = bf16x2_to_f16x2(w[u].z);
            w[u].w = bf16x2_to_f16x2(w[u].w);
            sts128(base + 4096u * u, w[u]);
          }
          fence_proxy_async_smem();  // this thread's writes are visible to the tensor cores' reads
          __syncwarp();
          if (lane == 0) mbar_arrive(&v_ready[vn % S]);
          ATTN_TR(22, j);  // this thread's share of V_j converted
        }
        ok = warp_wait(&s_full[t], g & 1, abort_v, kTimeoutNs);
        if (!ok) break;
        ATTN_TR(20, j);  // S_t(j) ready
        tc_fence_after();
        if constexpr (SPARSE) {
          // block-sparse mode: a tile no row of this warp sees (one only the other Q tile's
          // query block marks, or one past this tile's causal limit) has P = 0, written
          // without reading S or taking an exponential
          if (__all_sync(0xffffffffu, kmax < 0)) {
            uint32_t z[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) z[i] = 0u;
            tmem_st32(s_tmem + 64, z);
            tmem_st32(s_tmem + 96, z);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&p_full[t]);
            ATTN_TR(21, j);
            continue;
          }
        }
        uint32_t r[128];
        tmem_ld128_wait(s_tmem, r);
        if (masked) {
#pragma unroll
          for (int i = 0; i < 128; ++i) r[i] = (i > kmax) ? __float_as_uint(-INFINITY) : r[i];
        }
        const float m_in = m;  // the reference value the tile starts from
        // Row max of the tile; when it exceeds m, m moves kHeadroom above it.
        auto raise_to_tile_max = [&]() {
          float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
          for (int i = 0; i < 128; i += 8) {
            mx0 = max3f(mx0, __uint_as_float(r[i + 0]), __uint_as_float(r[i + 1]));
            mx1 = max3f(mx1, __uint_as_float(r[i + 2]), __uint_as_float(r[i + 3]));
            mx2 = max3f(mx2, __uint_as_float(r[i + 4]), __uint_as_float(r[i + 5]));
            mx3 = max3f(mx3, __uint_as_float(r[i + 6]), __uint_as_float(r[i + 7]));
          }
          const float m_tile = fmaxf(max3f(mx0, mx1, mx2), mx3) * c;
          if (m_tile > m) m = m_tile + kHeadroom;
        };
        // P = exp2(s * c - m): packed FMA and one ex2 per element, fp16 pairs into TMEM
        // columns 64-127 of S_t (P over keys 0-63, then 64-127), and the fp32 sum of P.
        // Keys 0-63 keep their fp32 P in r (in place of S); keys 64-127 keep their S in r.
        // The S of keys 0-63 also stays in TMEM columns 0-63 until the next S_t.
        uint64_t le0, le1;
        uint32_t pk0[32], pk1[32];
        auto exp_lo = [&]() {
          const float neg_m = (m == -INFINITY) ? 0.0f : -m;
          const uint64_t c2 = f2_pack(c, c);
          const uint64_t nm2 = f2_pack(neg_m, neg_m);
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            float x0, x1;
            f2_unpack(ffma2(f2_pack(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])), c2, nm2), x0, x1);
            const float p0 = ex2_approx(x0);
            const float p1 = ex2_approx(x1);
            r[2 * i] = __float_as_uint(p0);
            r[2 * i + 1] = __float_as_uint(p1);
            pk0[i] = pack_f16x2(p0, p1);
            if (i & 1)
              le1 = fadd2(le1, f2_pack(p0, p1));
            else
              le0 = fadd2(le0, f2_pack(p0, p1));
          }
          tmem_st32(s_tmem + 64, pk0);
        };
        auto exp_hi = [&]() {
          const float neg_m = (m == -INFINITY) ? 0.0f : -m;
          const uint64_t c2 = f2_pack(c, c);
          const uint64_t nm2 = f2_pack(neg_m, neg_m);
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            float x0, x1;
            f2_unpack(ffma2(f2_pack(__uint_as_float(r[64 + 2 * i]), __uint_as_float(r[64 + 2 * i + 1])), c2, nm2),
                      x0, x1);
            const float p0 = ex2_approx(x0);
            const float p1 = ex2_approx(x1);
            pk1[i] = pack_f16x2(p0, p1);
            if (i & 1)
              le1 = fadd2(le1, f2_pack(p0, p1));
            else
              le0 = fadd2(le0, f2_pack(p0, p1));
          }
          tmem_st32(s_tmem + 96, pk1);
        };
        auto mass = [&]() {
          float a0, a1, b0, b1;
          f2_unpack(le0, a0, a1);
          f2_unpack(le1, b0, b1);
          return (a0 + a1) + (b0 + b1);
        };
        // The row max only on a row's first tile, or while the row has seen no key.
        const bool first = __any_sync(0xffffffffu, j == 0 || m == -INFINITY);
        if (first) raise_to_tile_max();
        le0 = f2_pack(0.0f, 0.0f);
        le1 = le0;
        exp_lo();
        exp_hi();
        float tile_le = mass();
        // Rare: the tile's P mass passes fp16's largest value (NaN fails the comparison
        // too), so some P may have overflowed in fp16.  A finite mass up to 2^64 moves m
        // up by the exponent that brings it below 2^-8: keys 0-63 scale their fp32 P by
        // that power of two (exact), keys 64-127 redo theirs from S.  A larger or
        // non-finite mass takes the row max instead, with the S of keys 0-63 reloaded
        // from TMEM.  Both halves of P are then stored again.
        const bool slow = __any_sync(0xffffffffu, !(tile_le <= kF16Max));
        if (slow) {
          float sc = 1.0f;
          const bool huge = !(tile_le <= kScaleMassLimit);
          if (!(tile_le <= kF16Max) && !huge) {
            const int e = (__float_as_int(tile_le) >> 23) - 127;  // mass in [2^e, 2^(e+1)), e >= 15
            const int shift = e + 1 + kHeadroomBits;
            sc = __int_as_float((127 - shift) << 23);
            m += static_cast<float>(shift);
          }
          tmem_wait_st();  // the first pass's P stores have landed before they are overwritten
          if (__any_sync(0xffffffffu, huge)) {
            uint32_t s0[32], s1[32];
            tmem_ld32_wait(s_tmem, s0);
            tmem_ld32_wait(s_tmem + 32, s1);
            float mx = -INFINITY;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              s0[i] = (masked && i > kmax) ? __float_as_uint(-INFINITY) : s0[i];
              s1[i] = (masked && 32 + i > kmax) ? __float_as_uint(-INFINITY) : s1[i];
              mx = max3f(mx, __uint_as_float(s0[i]), __uint_as_float(s1[i]));
            }
#pragma unroll
            for (int i = 64; i < 128; i += 2) mx = max3f(mx, __uint_as_float(r[i]), __uint_as_float(r[i + 1]));
            mx *= c;
            if (huge && mx > m) m = mx + kHeadroom;
            const float neg_m = (m == -INFINITY) ? 0.0f : -m;
#pragma unroll
            for (int i = 0; i < 32; ++i) {  // huge rows: P of keys 0-63 again from S
              const float q0 = ex2_approx(fmaf(__uint_as_float(s0[i]), c, neg_m));
              const float q1 = ex2_approx(fmaf(__uint_as_float(s1[i]), c, neg_m));
              r[i] = huge ? __float_as_uint(q0) : r[i];
              r[32 + i] = huge ? __float_as_uint(q1) : r[32 + i];
            }
          }
          le0 = f2_pack(0.0f, 0.0f);
          le1 = le0;
          const uint64_t sc2 = f2_pack(sc, sc);
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            float p0, p1;
            f2_unpack(fmul2(f2_pack(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])), sc2), p0, p1);
            pk0[i] = pack_f16x2(p0, p1);
            if (i & 1)
              le1 = fadd2(le1, f2_pack(p0, p1));
            else
              le0 = fadd2(le0, f2_pack(p0, p1));
          }
          tmem_st32(s_tmem + 64, pk0);
          exp_hi();
          tile_le = mass();
        }
        // m moved: bring l, l_exact and (past the item's first tile) O_t to the new m.
        // O_t can be rewritten here: P.V_t(j-1) completed before S_t(j), whose commit came after it.
        const float alpha = (m == m_in) ? 1.0f : ex2_approx(m_in - m);
        if ((first || slow) && __any_sync(0xffffffffu, alpha != 1.0f)) {
          l *= alpha;
          l_exact *= alpha;
          if (j > 0) {
            const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll
            for (int cb = 0; cb < (C::kPvN + 31) / 32; ++cb) {  // O and, at D = 64, the row-sum columns
              uint32_t o[32];
              tmem_ld32_wait(o_tmem + cb * 32, o);
#pragma unroll
              for (int i = 0; i < 32; i += 2) {
                float x0, x1;
                f2_unpack(fmul2(f2_pack(__uint_as_float(o[i]), __uint_as_float(o[i + 1])), a2), x0, x1);
                o[i] = __float_as_uint(x0);
                o[i + 1] = __float_as_uint(x1);
              }
              tmem_st32(o_tmem + cb * 32, o);
            }
          }
        }
        l_exact += tile_le;
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&p_full[t]);
        ATTN_TR(21, j);  // P_t(j) handed to the MMA
        if constexpr (!C::kTensorRowSum) {  // the sum of the fp16-rounded P, after the hand-off
          float q0 = 0.0f, q1 = 0.0f, q2 = 0.0f, q3 = 0.0f;
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            add_f16x2_to_f32(q0, q1, pk0[i]);
            add_f16x2_to_f32(q2, q3, pk0[i + 1]);
            add_f16x2_to_f32(q0, q1, pk1[i]);
            add_f16x2_to_f32(q2, q3, pk1[i + 1]);
          }
          l += (q0 + q1) + (q2 + q3);
        }
      }
      if (!ok) {
        if (lane == 0) record_abort(abort_v, kSiteSoftmax);
        break;
      }

      // ---- epilogue: O = O_acc / l in bf16, LSE = (m + log2 l_exact) * ln 2.  O goes
      // through a 128-B-swizzled staging tile in shared memory and out with one TMA
      // store per 64 columns (coalesced; rows past Sq are clipped by the tensor map).
      ok = warp_wait(&o_final[t], n_done & 1, abort_v, kTimeoutNs);
      if (!ok) {
        if (lane == 0) record_abort(abort_v, kSiteEpilogue);
        break;
      }
      const uint32_t e_idx = n_done++;  // this Q tile's epilogue count (staging hand-off phase)
      tc_fence_after();
      uint32_t o[D];
      if constexpr (D == 128) {
        tmem_ld128_wait(o_tmem, o);
      } else {
        uint32_t lo[32], hi[32];
        tmem_ld32_wait(o_tmem, lo);
        tmem_ld32_wait(o_tmem + 32, hi);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          o[i] = lo[i];
          o[32 + i] = hi[i];
        }
        l = __uint_as_float(tmem_ld1_wait(o_tmem + D));  // rounded-P row sum from the tensor cores
      }
      tc_fence_before();
      mbar_arrive(&o_empty[t]);  // O_t may now be overwritten by the next item's first P.V
      ATTN_TR(23, x);  // O_t read out of TMEM
      const bool any_key = l > 0.0f;
      const float inv_l = any_key ? 1.0f / l : 0.0f;
      if (SPLIT) {  // fp32 partial O (normalised by this range's l) and partial LSE, for the merge
        if (live) {
          const uint64_t s2 = f2_pack(inv_l, inv_l);
          float4* dst = reinterpret_cast<float4*>(p.o_part + prow * D);
#pragma unroll
          for (int v4 = 0; v4 < D / 4; ++v4) {
            float x0, x1, x2, x3;
            f2_unpack(fmul2(f2_pack(__uint_as_float(o[4 * v4]), __uint_as_float(o[4 * v4 + 1])), s2), x0, x1);
            f2_unpack(fmul2(f2_pack(__uint_as_float(o[4 * v4 + 2]), __uint_as_float(o[4 * v4 + 3])), s2), x2, x3);
            dst[v4] = make_float4(x0, x1, x2, x3);
          }
          p.lse_part[prow] = any_key ? (m + lg2_approx(l_exact)) * 0.69314718055994531f : -INFINITY;
        }
        continue;
      }
      // the staging buffer: with one buffer the Q tiles take turns (tile 0, then tile 1, per item)
      const int sb = (C::kStageBufs == 1) ? 0 : t;
      uint8_t* stage = st_s + sb * C::kStageBytes;
      if (C::kStageBufs == 1) {
        if (t == 0) {
          if (e_idx > 0) ok = warp_wait(&stage_rel[1], (e_idx - 1) & 1, abort_v, kTimeoutNs);
        } else {
          ok = warp_wait(&stage_rel[0], e_idx & 1, abort_v, kTimeoutNs);
        }
      } else if (e_idx > 0) {
        ok = warp_wait(&stage_rel[t], (e_idx - 1) & 1, abort_v, kTimeoutNs);
      }
      if (!ok) {
        if (lane == 0) record_abort(abort_v, kSiteEpilogue);
        break;
      }
      {
        const int r = quarter * 32 + lane;  // row within the Q tile
        const uint64_t s2 = f2_pack(inv_l, inv_l);
#pragma unroll
        for (int ch = 0; ch < D / 8; ++ch) {  // 16-byte chunks of the row
          uint32_t w[4];
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            float x0, x1;
            const int e = ch * 8 + 2 * h;
            f2_unpack(fmul2(f2_pack(__uint_as_float(o[e]), __uint_as_float(o[e + 1])), s2), x0, x1);
            w[h] = pack_bf16x2(x0, x1);
          }
          const int cb = ch / 8, cc = ch % 8;
          uint4* dst = reinterpret_cast<uint4*>(stage + cb * (BM * 128) + r * 128 + ((cc ^ (r & 7)) << 4));
          *dst = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
      fence_proxy_async_smem();  // this thread's staged row is visible to the TMA store
      mbar_arrive(&stage_full[t]);  // the store warp writes the tile out
      ATTN_TR(24, x);  // O_t staged
      if (live) *lrow = any_key ? (m + lg2_approx(l_exact)) * 0.69314718055994531f : -INFINITY;
    }
    ATTN_TR_DONE();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ----------------------------------------------------------------------------
// host side
// ----------------------------------------------------------------------------
thread_local cudaError_t t_last_cuda_error = cudaSuccess;

int cuda_fail(cudaError_t e) {
  t_last_cuda_error = e;
  return ATTN_ERR_CUDA;
}

constexpr int kMaxDevices = 64;
std::atomic<unsigned int> g_launch_seq{0};   // picks each direct launch's schedule counter
std::atomic<unsigned int> g_capture_seq{0};  // picks each captured launch's schedule counter
std::mutex g_dev_mutex;
int g_dev_state[kMaxDevices];  // 0 unknown, 1 ready, -1 unsupported
int g_dev_sms[kMaxDevices];    // streaming multiprocessors per device
int64_t g_dev_l2[kMaxDevices];  // L2 bytes per device

// Capability check and kernel attributes, once per device.
int prepare_device(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  if (g_dev_state[dev] == 1) return ATTN_OK;
  if (g_dev_state[dev] == -1) return ATTN_ERR_UNSUPPORTED_DEVICE;
  int major = 0, minor = 0;
  cudaError_t e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (major != 10 || minor != 3) {
    g_dev_state[dev] = -1;
    return ATTN_ERR_UNSUPPORTED_DEVICE;
  }
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(e);
  g_dev_sms[dev] = sms;
  int l2 = 0;
  e = cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev);
  if (e != cudaSuccess) return cuda_fail(e);
  g_dev_l2[dev] = l2;
  const void* k128[] = {reinterpret_cast<const void*>(attn_fwd_kernel<128, false, false>),
                        reinterpret_cast<const void*>(attn_fwd_kernel<128, true, false>),
                        reinterpret_cast<const void*>(attn_fwd_kernel<128, false, true>),
                        reinterpret_cast<const void*>(attn_fwd_kernel<128, false, false, true>),
                        reinterpret_cast<const void*>(attn_fwd_kernel<128, false, false, false, true>),
                        reinterpret_cast<const void*>(attn_fwd_kernel<128, false, true, false, true>),
                        reinterpret_cast<const void*>(attn_fwd_kernel<128, false, false, true, true>)};
  const void* k64[] = {reinterpret_cast<const void*>(attn_fwd_kernel<64, false, false>),
                       reinterpret_cast<const void*>(attn_fwd_kernel<64, true, false>),
                       reinterpret_cast<const void*>(attn_fwd_kernel<64, false, true>),
                       reinterpret_cast<const void*>(attn_fwd_kernel<64, false, false, true>),
                       reinterpret_cast<const void*>(attn_fwd_kernel<64, false, false, false, true>),
                       reinterpret_cast<const void*>(attn_fwd_kernel<64, false, true, false, true>),
                       reinterpret_cast<const void*>(attn_fwd_kernel<64, false, false, true, true>)};
  for (const void* f : k128)
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<128>::kSmemBytes);
  for (const void* f : k64)
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<64>::kSmemBytes);
  if (e != cudaSuccess) return cuda_fail(e);
  if (!attn_host::encode_tiled_fn()) return ATTN_ERR_TENSOR_MAP;
  g_dev_state[dev] = 1;
  return ATTN_OK;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  if (na == 0 || nb == 0) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + nb && b0 < a0 + na;
}

bool misaligned(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) != 0; }

constexpr int kMaxSplits = 256;

// Merge of split-key partials (split-key mode): one warp per query row.
//   LSE = ln sum_r exp(LSE_r);  O = sum_r exp(LSE_r - LSE) O_r   (rows whose every LSE_r is -inf: O = 0)
// The weights are the exact probability mass of each key range; each O_r is
// already normalised within its range.
template <int D>
__global__ void __launch_bounds__(256) attn_merge_kernel(const float* __restrict__ o_part,
                                                         const float* __restrict__ lse_part,
                                                         __nv_bfloat16* __restrict__ o, float* __restrict__ lse,
                                                         int64_t rows, int n_splits) {
  constexpr int kPerLane = D / 32;  // 4 (D = 128) or 2 (D = 64) consecutive columns per lane
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  if (row >= rows) return;
  float mx = -INFINITY;
  for (int r = 0; r < n_splits; ++r) mx = fmaxf(mx, lse_part[r * rows + row]);
  float acc[kPerLane];
#pragma unroll
  for (int i = 0; i < kPerLane; ++i) acc[i] = 0.0f;
  float total = 0.0f;
  if (mx != -INFINITY) {
    for (int r = 0; r < n_splits; ++r) {
      const float w = expf(lse_part[r * rows + row] - mx);
      total += w;
      const float* src = o_part + (r * rows + row) * D + lane * kPerLane;
#pragma unroll
      for (int i = 0; i < kPerLane; ++i) acc[i] += w * src[i];
    }
  }
  const float inv = total > 0.0f ? 1.0f / total : 0.0f;
  __nv_bfloat16* dst = o + row * D + lane * kPerLane;
#pragma unroll
  for (int i = 0; i < kPerLane; i += 2) {
    const uint32_t w2 = pack_bf16x2(acc[i] * inv, acc[i + 1] * inv);
    *reinterpret_cast<uint32_t*>(dst + i) = w2;
  }
  if (lane == 0) lse[row] = mx == -INFINITY ? -INFINITY : mx + logf(total);
}

// Bytes of the split-key workspace: fp32 partial O, then (256-byte aligned) fp32 partial LSE.
size_t splitkv_bytes(int64_t rows, int D, int n_splits, size_t* lse_offset) {
  const size_t o_bytes = static_cast<size_t>(n_splits) * rows * D * 4;
  const size_t off = (o_bytes + 255) & ~static_cast<size_t>(255);
  if (lse_offset) *lse_offset = off;
  return off + static_cast<size_t>(n_splits) * rows * 4;
}

// Everything a launch needs, after the host-side checks.
struct Launch {
  CUtensorMap tq, tk, tv, to;
  Params prm;
  int grid = 0;
  int dev = 0;
  bool empty = false;  // B == 0 or Sq == 0: nothing to do
  bool grouped = false;  // dense mode: items in the grouped order (see item_at)
};

int prepare_launch(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int Sq,
                   int Sk, int D, int causal, float scale, int n_splits, cudaStream_t stream, Launch* L) {
  // ---- argument checks (host only, before any CUDA call)
  if (B < 0 || Sq < 0 || Sk < 0 || Hq < 1 || Hkv < 1) return ATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return ATTN_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (causal < 0 || causal > 2) return ATTN_ERR_INVALID_ARG;
  if (!(std::isfinite(scale) && scale > 0.0f)) return ATTN_ERR_INVALID_ARG;  // masking relies on scale > 0
  if (n_splits < 1 || n_splits > kMaxSplits) return ATTN_ERR_INVALID_ARG;
  const int64_t q_elems = static_cast<int64_t>(B) * Hq * Sq * D;
  const int64_t kv_elems = static_cast<int64_t>(B) * Hkv * Sk * D;
  const int64_t rows = static_cast<int64_t>(B) * Hq * Sq;
  if (static_cast<int64_t>(B) * Hq > INT32_MAX || static_cast<int64_t>(B) * Hkv > INT32_MAX)
    return ATTN_ERR_INVALID_ARG;
  L->empty = (B == 0 || Sq == 0);
  if (L->empty) return ATTN_OK;  // nothing to compute
  const int64_t n_qblocks = (Sq + ROWS_PER_ITEM - 1) / ROWS_PER_ITEM;
  const int64_t items = static_cast<int64_t>(B) * Hq * n_qblocks * n_splits;
  if (items > INT32_MAX) return ATTN_ERR_INVALID_ARG;
  if (!q || !o || !lse) return ATTN_ERR_NULL_PTR;
  if (Sk > 0 && (!k || !v)) return ATTN_ERR_NULL_PTR;
  if (misaligned(q) || misaligned(o) || misaligned(lse)) return ATTN_ERR_MISALIGNED;
  if (Sk > 0 && (misaligned(k) || misaligned(v))) return ATTN_ERR_MISALIGNED;
  const size_t qb = static_cast<size_t>(q_elems) * 2, kvb = static_cast<size_t>(kv_elems) * 2;
  const size_t lb = static_cast<size_t>(rows) * 4;
  if (overlaps(o, qb, q, qb) || overlaps(o, qb, k, kvb) || overlaps(o, qb, v, kvb) || overlaps(o, qb, lse, lb) ||
      overlaps(lse, lb, q, qb) || overlaps(lse, lb, k, kvb) || overlaps(lse, lb, v, kvb))
    return ATTN_ERR_INVALID_ARG;

  // ---- device
  cudaError_t e = cudaGetDevice(&L->dev);
  if (e != cudaSuccess) return cuda_fail(e);
  const int st = prepare_device(L->dev);
  if (st != ATTN_OK) return st;

  // ---- TMA maps: Q, O [B*Hq][Sq][D], K/V [B*Hkv][Sk][D]; boxes of 64 columns x 128 rows
  if (!attn_host::encode_bf16_rows(&L->tq, q, D, Sq, static_cast<uint64_t>(B) * Hq, BM)) return ATTN_ERR_TENSOR_MAP;
  if (!attn_host::encode_bf16_rows(&L->to, o, D, Sq, static_cast<uint64_t>(B) * Hq, BM)) return ATTN_ERR_TENSOR_MAP;
  if (Sk > 0) {
    if (!attn_host::encode_bf16_rows(&L->tk, k, D, Sk, static_cast<uint64_t>(B) * Hkv, BN))
      return ATTN_ERR_TENSOR_MAP;
    if (!attn_host::encode_bf16_rows(&L->tv, v, D, Sk, static_cast<uint64_t>(B) * Hkv, BN))
      return ATTN_ERR_TENSOR_MAP;
  } else {
    L->tk = L->tq;  // never read: every row is fully masked and no key tile is loaded
    L->tv = L->tq;
  }

  Params& prm = L->prm;
  prm.o = static_cast<__nv_bfloat16*>(o);
  prm.lse = lse;
  prm.Hq = Hq;
  prm.Hkv = Hkv;
  prm.G = Hq / Hkv;
  prm.Sq = Sq;
  prm.Sk = Sk;
  prm.causal = causal != 0;
  prm.diag = causal == 1 ? Sk - Sq : 0;
  prm.n_qblocks = static_cast<int>(n_qblocks);
  prm.BH = B * Hq;
  prm.n_items = static_cast<int>(items);
  prm.c = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634074);
  prm.n_splits = n_splits;
  prm.o_part = nullptr;
  prm.lse_part = nullptr;
  {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    e = cudaStreamIsCapturing(stream, &cs);
    if (e != cudaSuccess) return cuda_fail(e);
    prm.sched_slot = (cs == cudaStreamCaptureStatusActive)
                         ? kEagerSlots + static_cast<int>(g_capture_seq.fetch_add(1, std::memory_order_relaxed) %
                                                          kCaptureSlots)
                         : static_cast<int>(g_launch_seq.fetch_add(1, std::memory_order_relaxed) % kEagerSlots);
  }
  prm.mask = nullptr;
  prm.order = nullptr;
  prm.order_heads = 1;
  prm.order_len = 0;
  prm.mask_heads = 1;
  prm.mask_words = 0;
  prm.n_qtiles = static_cast<int>((Sq + BM - 1) / BM);
  // persistent: one CTA per SM (shared memory and TMEM allow no second), never more CTAs than items
  L->grid = static_cast<int>(items < g_dev_sms[L->dev] ? items : g_dev_sms[L->dev]);
  // The grouped item order when K and V of all kv heads do not fit in L2: in the heads-fastest order a kv
  // head's items fall into different waves, so its K and V tiles come from HBM about once per wave (long
  // context: 7.65 GB read per launch instead of 0.82 GB).  When they fit, the heads-fastest order keeps the
  // whole list heaviest first, which the causal shapes need (the grouped order is heaviest first only within
  // a kv head).
  {
    const int64_t per = static_cast<int64_t>(Hq / Hkv) * n_qblocks;  // items of one kv head
    const int64_t kv_bytes = 2 * kv_elems * 2;
    L->grouped = n_splits == 1 && per >= 2 && kv_bytes > g_dev_l2[L->dev];
    // ATTN_FWD_ITEM_ORDER=heads or =grouped overrides the choice (the results are the same bit for bit)
    const char* order = std::getenv("ATTN_FWD_ITEM_ORDER");
    if (order && std::strcmp(order, "heads") == 0) L->grouped = false;
    if (order && std::strcmp(order, "grouped") == 0) L->grouped = n_splits == 1;
  }
  return ATTN_OK;
}

template <int D, bool SPLIT, bool SPARSE = false, bool ORDERED = false, bool GROUPED = false>
int launch(const Launch& L, cudaStream_t stream) {
  attn_fwd_kernel<D, SPLIT, SPARSE, ORDERED, GROUPED><<<L.grid, kThreads, Cfg<D>::kSmemBytes, stream>>>(
      L.tq, L.tk, L.tv, L.to, L.prm);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}

// The dense kernel in the item order prepare_launch chose.
int launch_dense(const Launch& L, int D, cudaStream_t stream) {
  if (L.grouped)
    return D == 128 ? launch<128, false, false, false, true>(L, stream) : launch<64, false, false, false, true>(L, stream);
  return D == 128 ? launch<128, false>(L, stream) : launch<64, false>(L, stream);
}

template <int D>
int launch_merge(const Launch& L, int64_t rows, cudaStream_t stream) {
  const int64_t blocks = (rows + 7) / 8;
  attn_merge_kernel<D><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(L.prm.o_part, L.prm.lse_part, L.prm.o,
                                                                           L.prm.lse, rows, L.prm.n_splits);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}

// Split-key forward with the partials in `ws` (device memory, at least splitkv_bytes).
// One range is the plain forward: the merge of a single partial multiplies it by
// exactly 1, so the plain kernel writes the same values without the partials.
int run_splitkv(const Launch& L0, void* ws, int64_t rows, int D, cudaStream_t stream) {
  if (L0.prm.n_splits == 1) return launch_dense(L0, D, stream);
  Launch L = L0;
  size_t lse_off = 0;
  splitkv_bytes(rows, D, L.prm.n_splits, &lse_off);
  L.prm.o_part = static_cast<float*>(ws);
  L.prm.lse_part = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + lse_off);
  int st = D == 128 ? launch<128, true>(L, stream) : launch<64, true>(L, stream);
  if (st != ATTN_OK) return st;
  return D == 128 ? launch_merge<128>(L, rows, stream) : launch_merge<64>(L, rows, stream);
}

}  // namespace

// Fixed scratch for attn_fwd_splitkv_noalloc: the split-key partials of callers
// that cannot allocate device memory.  Every device that loads this library
// holds these 32 MiB until the process exits.  Host code only uses the name to
// look up the device address (cudaGetSymbolAddress), once per CUDA context.
constexpr size_t kNoAllocScratchBytes = size_t{32} << 20;
static __device__ __align__(256) unsigned char g_splitkv_scratch[kNoAllocScratchBytes];

namespace {

std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices];                // device address of g_splitkv_scratch, per device
unsigned long long g_scratch_ctx[kMaxDevices];    // ... and the id of the context it was looked up in

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Unique id of the calling thread's current context (ids are never reused within
// a process, so a context created after a cudaDeviceReset gets a new one); false
// when the driver does not provide it.
bool current_context_id(unsigned long long* id) {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  CUcontext ctx = nullptr;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
  return get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of the fixed scratch on `dev` (the current device), looked up on
// the first call in each context: an address from an earlier context (before a
// cudaDeviceReset, say) is never reused.
int noalloc_scratch(int dev, void** out) {
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED_DEVICE;
  unsigned long long ctx = 0;
  const bool have_ctx = current_context_id(&ctx);
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_addr[dev] == nullptr || !have_ctx || g_scratch_ctx[dev] != ctx) {
    void* ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_splitkv_scratch);
    if (e != cudaSuccess) return cuda_fail(e);
    g_scratch_addr[dev] = ptr;
    g_scratch_ctx[dev] = ctx;
  }
  *out = g_scratch_addr[dev];
  return ATTN_OK;
}

}  // namespace

extern "C" {

int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int Sq,
             int Sk, int D, int causal, float scale, cudaStream_t stream) {
  Launch L;
  const int st = prepare_launch(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, causal, scale, 1, stream, &L);
  if (st != ATTN_OK || L.empty) return st;
  return launch_dense(L, D, stream);
}

size_t attn_fwd_splitkv_workspace_size(int B, int Hq, int Sq, int D, int n_splits) {
  if (B < 0 || Hq < 0 || Sq < 0 || (D != 64 && D != 128) || n_splits < 1 || n_splits > kMaxSplits) return 0;
  return splitkv_bytes(static_cast<int64_t>(B) * Hq * Sq, D, n_splits, nullptr);
}

int attn_fwd_splitkv_suggest(int B, int Hq, int Sq, int Sk, int D, int causal) {
  if (B < 1 || Hq < 1 || Sq < 1 || Sk < 1 || (D != 64 && D != 128) || causal < 0 || causal > 2) return 1;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || prepare_device(dev) != ATTN_OK) return 1;
  const double sms = g_dev_sms[dev];
  // Key tiles of every 256-row query block (the work items of one (batch, head)), as the kernel counts them.
  const int64_t n_qblocks = (Sq + ROWS_PER_ITEM - 1) / ROWS_PER_ITEM;
  const int64_t diag = causal == 1 ? static_cast<int64_t>(Sk) - Sq : 0;
  double tiles_sum = 0.0, tiles_max = 0.0;
  for (int64_t qb = 0; qb < n_qblocks; ++qb) {
    const int64_t last_row = std::min<int64_t>((qb + 1) * ROWS_PER_ITEM, Sq) - 1;
    const int64_t kv_end = causal ? std::min<int64_t>(Sk, last_row + diag + 1) : Sk;
    const double n = kv_end > 0 ? static_cast<double>((kv_end + BN - 1) / BN) : 0.0;
    tiles_sum += n;
    tiles_max = std::max(tiles_max, n);
  }
  const double items = static_cast<double>(B) * Hq * n_qblocks;
  if (tiles_max < 8.0) return 1;
  // Cost model of a launch, calibrated on GB300: a key tile of an item takes t_step, an
  // item's start and end t_item; the CTAs run the items in waves (ceil(items / SMs) when
  // the items are about equal, at least the largest one); the partials cost (D + 1)
  // fp32 per row and range written and read again, plus the output, at an effective
  // 4 TB/s, and the merge a launch of its own.
  const double t_step = D == 128 ? 1.55e-6 : 1.2e-6, t_item = 2.5e-6;
  const double rows = static_cast<double>(B) * Hq * Sq;
  const double mean_tiles = tiles_sum / n_qblocks;
  const int s_max = static_cast<int>(std::min<double>(kMaxSplits, tiles_max / 4.0));  // >= 4 key tiles per range
  int best = 1;
  double best_cost = 0.0;
  for (int s = 1; s <= s_max; ++s) {
    const double waves = std::ceil(items * s / sms);
    const double makespan = std::max(waves * (mean_tiles / s * t_step + t_item), tiles_max / s * t_step + t_item);
    const double merge = s > 1 ? 3e-6 + rows * ((D + 1) * 4.0 * s * 2.0 + D * 2.0 + 4.0) / 4e12 : 0.0;
    const double cost = makespan + merge;
    if (s == 1 || cost < best_cost * 0.97) {  // a split must gain at least 3 % to be taken
      best = s;
      best_cost = cost;
    }
  }
  return best;
}

int attn_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                     int Sq, int Sk, int D, int causal, float scale, int n_splits, void* workspace,
                     size_t workspace_bytes, cudaStream_t stream) {
  Launch L;
  const int st = prepare_launch(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, causal, scale, n_splits, stream, &L);
  if (st != ATTN_OK || L.empty) return st;
  const int64_t rows = static_cast<int64_t>(B) * Hq * Sq;
  if (!workspace) return ATTN_ERR_NULL_PTR;
  if (misaligned(workspace)) return ATTN_ERR_MISALIGNED;
  const size_t need = splitkv_bytes(rows, D, n_splits, nullptr);
  if (workspace_bytes < need) return ATTN_ERR_INVALID_ARG;
  const size_t qb = static_cast<size_t>(rows) * D * 2;
  const size_t kvb = static_cast<size_t>(B) * Hkv * Sk * D * 2;
  if (overlaps(workspace, need, q, qb) || overlaps(workspace, need, k, kvb) || overlaps(workspace, need, v, kvb) ||
      overlaps(workspace, need, o, qb) || overlaps(workspace, need, lse, static_cast<size_t>(rows) * 4))
    return ATTN_ERR_INVALID_ARG;
  return run_splitkv(L, workspace, rows, D, stream);
}

size_t attn_fwd_block_mask_words(int B, int mask_heads, int Sq, int Sk) {
  if (B < 0 || mask_heads < 1 || Sq < 0 || Sk < 0) return 0;
  const int64_t kblocks = (static_cast<int64_t>(Sk) + BN - 1) / BN;
  const int64_t qblocks = (static_cast<int64_t>(Sq) + BM - 1) / BM;
  return static_cast<size_t>(B) * mask_heads * qblocks * ((kblocks + 31) / 32);
}

int attn_fwd_blocksparse(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                         int Sq, int Sk, int D, int causal, float scale, const uint32_t* block_mask, int mask_heads,
                         cudaStream_t stream) {
  // the mask's own checks (host only, before any CUDA call), then the common ones
  if (Hq < 1 || (mask_heads != 1 && mask_heads != Hq)) return ATTN_ERR_INVALID_ARG;
  const size_t words = (B > 0 && Sq > 0 && Sk > 0) ? attn_fwd_block_mask_words(B, mask_heads, Sq, Sk) : 0;
  if (words > 0) {
    if (!block_mask) return ATTN_ERR_NULL_PTR;
    if ((reinterpret_cast<uintptr_t>(block_mask) & 3u) != 0) return ATTN_ERR_MISALIGNED;
    if (D > 0) {
      const size_t mb = words * 4;
      const size_t qb = static_cast<size_t>(B) * Hq * Sq * D * 2, lb = static_cast<size_t>(B) * Hq * Sq * 4;
      if (overlaps(block_mask, mb, o, qb) || overlaps(block_mask, mb, lse, lb)) return ATTN_ERR_INVALID_ARG;
    }
  }
  Launch L;
  const int st = prepare_launch(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, causal, scale, 1, stream, &L);
  if (st != ATTN_OK || L.empty) return st;
  L.prm.mask = block_mask;
  L.prm.mask_heads = mask_heads;
  L.prm.mask_words = static_cast<int>(((static_cast<int64_t>(Sk) + BN - 1) / BN + 31) / 32);
  if (L.grouped)
    return D == 128 ? launch<128, false, true, false, true>(L, stream) : launch<64, false, true, false, true>(L, stream);
  return D == 128 ? launch<128, false, true>(L, stream) : launch<64, false, true>(L, stream);
}

size_t attn_fwd_tile_order_entries(int B, int order_heads, int Sq, int Sk) {
  if (B < 0 || order_heads < 1 || Sq < 0 || Sk < 0) return 0;
  const int64_t kblocks = (static_cast<int64_t>(Sk) + BN - 1) / BN;
  const int64_t qblocks = (static_cast<int64_t>(Sq) + ROWS_PER_ITEM - 1) / ROWS_PER_ITEM;
  return static_cast<size_t>(B) * order_heads * qblocks * kblocks;
}

int attn_fwd_ordered(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv, int Sq,
                     int Sk, int D, int causal, float scale, const int32_t* tile_order, int order_heads,
                     cudaStream_t stream) {
  // the order's own checks (host only, before any CUDA call), then the common ones
  if (Hq < 1 || (order_heads != 1 && order_heads != Hq)) return ATTN_ERR_INVALID_ARG;
  const size_t entries = (B > 0 && Sq > 0 && Sk > 0) ? attn_fwd_tile_order_entries(B, order_heads, Sq, Sk) : 0;
  if (entries > 0) {
    if (!tile_order) return ATTN_ERR_NULL_PTR;
    if ((reinterpret_cast<uintptr_t>(tile_order) & 3u) != 0) return ATTN_ERR_MISALIGNED;
    if (D > 0) {
      const size_t ob = entries * 4;
      const size_t qb = static_cast<size_t>(B) * Hq * Sq * D * 2, lb = static_cast<size_t>(B) * Hq * Sq * 4;
      if (overlaps(tile_order, ob, o, qb) || overlaps(tile_order, ob, lse, lb)) return ATTN_ERR_INVALID_ARG;
    }
  }
  Launch L;
  const int st = prepare_launch(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, causal, scale, 1, stream, &L);
  if (st != ATTN_OK || L.empty) return st;
  L.prm.order = tile_order;
  L.prm.order_heads = order_heads;
  L.prm.order_len = static_cast<int>((static_cast<int64_t>(Sk) + BN - 1) / BN);
  if (L.grouped)
    return D == 128 ? launch<128, false, false, true, true>(L, stream) : launch<64, false, false, true, true>(L, stream);
  return D == 128 ? launch<128, false, false, true>(L, stream) : launch<64, false, false, true>(L, stream);
}

int attn_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                             int Hkv, int Sq, int Sk, int D, int causal, float scale, int n_splits,
                             cudaStream_t stream) {
  Launch L;
  const int st = prepare_launch(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, causal, scale, n_splits, stream, &L);
  if (st != ATTN_OK || L.empty) return st;
  const int64_t rows = static_cast<int64_t>(B) * Hq * Sq;
  if (splitkv_bytes(rows, D, n_splits, nullptr) > kNoAllocScratchBytes) return ATTN_ERR_INVALID_ARG;
  void* scratch = nullptr;
  const int sst = noalloc_scratch(L.dev, &scratch);
  if (sst != ATTN_OK) return sst;
  // Every partial row is written by the first kernel before the merge reads it,
  // so what an earlier call left in the scratch is never read: nothing to clear.
  return run_splitkv(L, scratch, rows, D, stream);
}

#ifdef ATTN_TRACE
int attn_fwd_trace_read(void* dst, size_t dst_bytes, int* ctas, int* roles, int* events) {
  if (ctas) *ctas = kTraceCtas;
  if (roles) *roles = kTraceRoles;
  if (events) *events = kTraceEvents;
  const size_t n_bytes = sizeof(unsigned int) * kTraceCtas * kTraceRoles;
  const size_t r_bytes = sizeof(TraceRec) * static_cast<size_t>(kTraceCtas) * kTraceRoles * kTraceEvents;
  if (!dst) return ATTN_ERR_NULL_PTR;
  if (dst_bytes < n_bytes + r_bytes) return ATTN_ERR_INVALID_ARG;
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(dst, g_trace_n, n_bytes);
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(static_cast<uint8_t*>(dst) + n_bytes, g_trace, r_bytes);
  static const unsigned int zeros[kTraceCtas * kTraceRoles] = {};  // the next launch starts from empty counts
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_trace_n, zeros, n_bytes);
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}
#endif

const char* attn_fwd_strerror(int status) {
  switch (status) {
    case ATTN_OK: return "success";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_NULL_PTR: return "null pointer";
    case ATTN_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case ATTN_ERR_UNSUPPORTED_DEVICE: return "device is not compute capability 10.3 (sm_103a)";
    case ATTN_ERR_CUDA: return cudaGetErrorString(t_last_cuda_error);
    case ATTN_ERR_DEVICE_TIMEOUT: return "a kernel wait ran out of time; the kernel unwound";
    case ATTN_ERR_TENSOR_MAP: return "TMA tensor map rejected by the driver";
    default: return "unknown status";
  }
}

int attn_fwd_version(void) { return 100; }  // 0.1.0

int attn_fwd_debug_status(cudaStream_t stream, int* site) {
  if (site) *site = 0;
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e);
  int value = 0;
  e = cudaMemcpyFromSymbol(&value, g_status, sizeof(int));
  if (e != cudaSuccess) return cuda_fail(e);
  if (value != 0) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_status, &zero, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e);
  }
  if (site) *site = value;
  return value == 0 ? ATTN_OK : ATTN_ERR_DEVICE_TIMEOUT;
}

}  // extern "C"
