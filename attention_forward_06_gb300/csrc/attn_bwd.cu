// attn_bwd.cu -- backward of the exact attention forward pass for GB300 (sm_103a):
// the gradients of O = softmax(scale * Q K^T + mask) V with respect to Q, K and V
// for an upstream gradient dO, from the forward's saved LSE (the softmax with a
// closed-form log-sum-exp normaliser of page "AdaSplash-2: Faster Differentiable
// Sparse Attention", technical summary section 1; its summary notes that the
// backward pass, too, visits only the blocks it needs).  With P_ij recomputed as
// exp(scale q_i.k_j - LSE_i):
//     dV_j = sum_i P_ij dO_i,   dP_ij = dO_i . v_j,   D_i = dO_i . O_i,
//     dS_ij = P_ij (dP_ij - D_i),   dQ_i = scale sum_j dS_ij k_j,   dK_j = scale sum_i dS_ij q_i.
//
// Three kernels on the caller's stream:
//   attn_bwd_prep_kernel   -D_i = -dO_i . O_i and -LSE_i * log2(e) into the workspace
//                          (-inf for rows without keys and for padding rows, so their P is 0)
//   attn_bwd_dkdv_kernel   one (batch, kv head, 128-key tile) per work item: streams the
//                          query tiles of every query head of the group, with the keys in
//                          the TMEM lanes: S^T = K Q^T and dP^T = V dO^T (SS form), P^T and
//                          dS^T written back as bf16, then dV += P^T dO and dK += dS^T Q (TS
//                          form, A from TMEM) accumulate in TMEM across the whole item
//   attn_bwd_dq_kernel     one (batch, query head, 128-row tile) per item: S = Q K^T,
//                          dP = dO V^T, dS into TMEM, dQ += dS K
// The dK/dV kernel takes a step (a 128-row query tile) in two 64-wide halves held in
// two TMEM regions, warpgroup r (warps 4r .. 4r+3, one thread per TMEM lane) computing
// half r while the tensor cores run the other half's products; the dQ kernel computes a
// step's S and dP 128 keys wide, alternating two S regions, and its warpgroups split
// the keys.  Warp 8 loads with TMA, warp 9 issues the tcgen05 MMAs, warps 10-11 idle;
// every wait is bounded as in the forward.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "attn_bwd.h"
#include "host_util.h"
#include "ptx.cuh"

using namespace attn;

namespace {

constexpr int BT = 128;  // query rows / keys per tile (MMA M)
constexpr int BH2 = 64;  // query rows of a half step (dK/dV: MMA N of S^T, dP^T), keys per warpgroup (dQ)
constexpr int kHalfBytes = BH2 * 128;  // byte offset of a tile's second half of rows in a 128-B-swizzled block
constexpr int kThreads = 384;          // three warpgroups
constexpr int kComputeWarps = 8;       // warpgroup r computes half r of every step
constexpr int kLoadWarp = 8;
constexpr int kMmaWarp = 9;            // warps 10 and 11 idle (they complete the third warpgroup)
constexpr uint32_t kRegsLaunch = 168;   // 65536 / 384
constexpr uint32_t kRegsCompute = 224;  // dQ kernel: warpgroups 0 and 1 ...
constexpr uint32_t kRegsOther = 56;     // ... and warpgroup 2
static_assert(256 * kRegsCompute + 128 * kRegsOther <= kThreads * kRegsLaunch, "register split exceeds the pool");
// dK/dV kernel: its producer and issuer spill at 56 registers (ptxas) with the epilogue's shuffles
constexpr uint32_t kRegsComputeKV = 216, kRegsOtherKV = 72;
static_assert(256 * kRegsComputeKV + 128 * kRegsOtherKV <= kThreads * kRegsLaunch, "register split exceeds the pool");
constexpr int kRing = 2;  // streamed Q/dO tile-pair slots of the dK/dV kernel
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kTimeoutNs = 4000000000ull;
constexpr uint64_t kDrainTimeoutNs = 500000000ull;
constexpr int kSiteProducer = 1, kSiteIssuer = 2, kSiteCompute = 3;

template <int D>
struct BCfg {
  static constexpr int kTileBytes = BT * D * 2;    // one 128-row bf16 tile
  static constexpr int kColBlockBytes = BT * 128;  // 64 columns x 128 rows, 128-B swizzled
  static constexpr int kVecBytes = BT * 4;         // 128 fp32 values
  static constexpr int kSlotBytes = 2 * kTileBytes + 2 * kVecBytes;
  static constexpr int kSmemBytes = 2 * kTileBytes + kRing * kSlotBytes + 1024;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

struct BParams {
  __nv_bfloat16* dq;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  const float* nlse2;   // [B*Hq][Sq_pad]: -LSE * log2(e), -inf where P must be 0
  const float* ndelta;  // [B*Hq][Sq_pad]: -dO . O
  int Hq, Hkv, G, Sq, Sk, Sq_pad;
  int causal, diag;  // key j visible to row i iff !causal or j <= i + diag
  int n_qt, n_kt;    // 128-row query tiles, 128-key tiles
  int BZ;            // B * Hkv (dK/dV items) ...
  int BH;            // ... and B * Hq (dQ items)
  int n_items;
  float c;      // scale * log2(e)
  float scale;
};

__device__ int g_bwd_status;

#ifdef ATTN_TRACE
// Timeline build (-DATTN_TRACE, off by default): lane 0 of each role of the dK/dV
// kernel (kernel 0) and the dQ kernel (kernel 1) records (%globaltimer, event,
// argument) at the points listed in attn_bwd_trace.h, in a fixed device array that
// attn_bwd_trace_read copies out.  Without the switch every trace point compiles to
// nothing.
constexpr int kTraceKernels = 2;    // dK/dV, dQ
constexpr int kTraceRoles = 4;      // producer, issuer, compute warpgroup 0, compute warpgroup 1
constexpr int kTraceEvents = 2048;  // per role and CTA; later events are counted but not kept
constexpr int kTraceCtas = 160;     // CTAs numbered past this are not recorded
struct TraceRec {
  unsigned long long t;
  unsigned int code;
  unsigned int arg;
};
__device__ TraceRec g_btrace[kTraceKernels * kTraceCtas * kTraceRoles * kTraceEvents];
__device__ unsigned int g_btrace_n[kTraceKernels * kTraceCtas * kTraceRoles];
struct Tracer {
  int slot;  // (kernel * kTraceCtas + CTA) * kTraceRoles + role, or -1 when not recording
  unsigned int n;
  __device__ __forceinline__ void rec(unsigned int code, unsigned int arg) {
    if (slot < 0) return;
    if (n < kTraceEvents) g_btrace[static_cast<size_t>(slot) * kTraceEvents + n] = TraceRec{global_timer_ns(), code, arg};
    ++n;
  }
  __device__ __forceinline__ void done() {
    if (slot >= 0) g_btrace_n[slot] = n;
  }
};
__device__ __forceinline__ int trace_slot(int kernel, int role, bool on) {
  return (on && blockIdx.x < kTraceCtas) ? (kernel * kTraceCtas + static_cast<int>(blockIdx.x)) * kTraceRoles + role
                                         : -1;
}
#define ATTN_TR_DECL(kernel, role, on) Tracer tr_{trace_slot((kernel), (role), (on)), 0u}
#define ATTN_TR(code, arg) tr_.rec((code), static_cast<unsigned int>(arg))
#define ATTN_TR_DONE() tr_.done()
#else
#define ATTN_TR_DECL(kernel, role, on) ((void)0)
#define ATTN_TR(code, arg) ((void)0)
#define ATTN_TR_DONE() ((void)0)
#endif

__device__ __forceinline__ uint8_t* align_1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~static_cast<uintptr_t>(1023));
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile uint32_t* abort_flag,
                                          uint64_t timeout_ns) {
  const bool ok = mbar_wait_bounded(bar, parity, abort_flag, timeout_ns);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void record_abort(volatile uint32_t* abort_flag, int site) {
  *abort_flag = 1;
  atomicCAS(&g_bwd_status, 0, site);
}

// Stores 32 rows of a warp, one row per lane (lane m holds its row's CH 16-byte chunks in
// w[0 .. 4 CH)), row m at base + m * stride; rows m >= live_rows are skipped.  A warp store
// of one 16-byte chunk per lane would touch 32 rows (32 cache lines); instead the chunks are
// transposed within each group of CH lanes (log2 CH butterfly stages of shuffles, each
// swapping one bit between lane and chunk index), after which lane CH g + q holds chunk q of
// rows CH g .. CH g + CH - 1, and each of the CH stores writes 32 / CH whole rows.
template <int CH>
__device__ __forceinline__ void store_warp_rows(uint32_t (&w)[4 * CH], uint8_t* base, int64_t stride, int live_rows,
                                                int lane) {
  const int q = lane % CH;
#pragma unroll
  for (int b = CH / 2; b >= 1; b /= 2) {
    const bool hi = (q & b) != 0;
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      if (c & b) continue;
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const uint32_t send = hi ? w[4 * c + h] : w[4 * (c ^ b) + h];
        const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, b);
        if (hi)
          w[4 * c + h] = recv;
        else
          w[4 * (c ^ b) + h] = recv;
      }
    }
  }
  const int m0 = lane - q;
#pragma unroll
  for (int k = 0; k < CH; ++k)
    if (m0 + k < live_rows)
      *reinterpret_cast<uint4*>(base + (m0 + k) * stride + 16 * q) =
          make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
}

// ---------------------------------------------------------------------------- prep
// Rows of B*Hq*Sq_pad, 32 / (D/8) per warp, each lane reading 16 bytes of O and of dO:
// -D_i = -sum_d dO[i,d] O[i,d] (fp32, from the bf16 tensors) and -LSE_i * log2(e); rows
// past Sq and rows without keys (LSE = -inf) get -inf, so their P is 0.  The values are
// stored negated so the kernels add them with packed FMAs.
template <int D>
__global__ void __launch_bounds__(256) attn_bwd_prep_kernel(const __nv_bfloat16* __restrict__ o,
                                                            const __nv_bfloat16* __restrict__ dout,
                                                            const float* __restrict__ lse, float* __restrict__ nlse2,
                                                            float* __restrict__ ndelta, int64_t BH, int Sq,
                                                            int Sq_pad) {
  constexpr int kLanesPerRow = D / 8;
  constexpr int kRowsPerWarp = 32 / kLanesPerRow;
  const int lane = threadIdx.x % 32, sub = lane % kLanesPerRow;
  const int64_t row =
      (static_cast<int64_t>(blockIdx.x) * 8 + threadIdx.x / 32) * kRowsPerWarp + lane / kLanesPerRow;
  const bool in = row < BH * Sq_pad;
  float acc = 0.0f, nl2 = -INFINITY;
  if (in) {
    const int64_t bh = row / Sq_pad;
    const int i = static_cast<int>(row % Sq_pad);
    if (i < Sq) {
      const int64_t r = bh * Sq + i;
      const uint4 a = reinterpret_cast<const uint4*>(o + r * D)[sub];
      const uint4 b = reinterpret_cast<const uint4*>(dout + r * D)[sub];
      const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        acc = fmaf(bf16lo_to_f32(av[e]), bf16lo_to_f32(bv[e]), acc);
        acc = fmaf(bf16hi_to_f32(av[e]), bf16hi_to_f32(bv[e]), acc);
      }
      const float L = lse[r];
      nl2 = (L == -INFINITY) ? -INFINITY : -L * 1.4426950408889634f;
    }
  }
#pragma unroll
  for (int off = kLanesPerRow / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (in && sub == 0) {
    nlse2[row] = nl2;
    ndelta[row] = -acc;
  }
  griddep_launch_dependents();  // the dK/dV kernel may start its set-up
}

// The k-th work item of this CTA.  Items are listed heaviest first and dealt in
// rounds of gridDim.x, forwards on even rounds and backwards on odd ones, so every
// CTA gets a similar amount of work (every role walks the same sequence).
__device__ __forceinline__ int item_of(int k) {
  const int c = static_cast<int>(blockIdx.x), G = static_cast<int>(gridDim.x);
  return k * G + ((k & 1) ? G - 1 - c : c);
}

// Query tiles [i0, n_qt) that see key tile j (none when i0 >= n_qt).
__device__ __forceinline__ int first_qtile(const BParams& p, int j) {
  if (!p.causal) return 0;
  const int first_row = BT * j - p.diag;  // row i sees key 128 j iff i + diag >= 128 j
  if (first_row <= 0) return 0;
  if (first_row >= p.Sq) return p.n_qt;
  return first_row / BT;
}

// ---------------------------------------------------------------------------- dK, dV
// Work item x: key tile j = x / (B*Hkv) (ascending: under a causal mask the
// heaviest first), kv slice z = x % (B*Hkv).  A step is one 128-row query tile of
// one query head of the group, taken in two halves of 64 rows; half r lives in
// TMEM region r (lane = key): S^T_r at columns [128 r, 128 r + 64), dP^T_r at
// [128 r + 64, 128 r + 128), and P^T_r, dS^T_r (bf16 pairs) are written over the
// first 32 columns of each.  dV [256, 256 + D) and dK [384, 384 + D) accumulate
// over the whole item.  Compute warpgroup r owns half r, so one half's
// exponentials run while the tensor cores work on the other half:
//   S_0(s) S_1(s) | dVdK_0(s) S_0(s+1) dVdK_1(s) S_1(s+1) | ...
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                         const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                         const BParams p) {
  using C = BCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_1024(smem_raw);
  uint8_t* k_s = smem;
  uint8_t* v_s = smem + C::kTileBytes;
  uint8_t* ring = smem + 2 * C::kTileBytes;  // slot: Q, dO, -lse2[128], -delta[128]
  __shared__ uint64_t kv_full, kv_empty, full[kRing], empty[kRing], st_full[2], pt_full[2], acc_full, acc_empty,
      drain;
  __shared__ uint32_t tmem_slot, abort_flag;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int nz = p.BZ;

  if (threadIdx.x == 0) {
    mbar_init(&kv_full, 1);
    mbar_init(&kv_empty, 1);
    for (int s = 0; s < kRing; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int r = 0; r < 2; ++r) {
      mbar_init(&st_full[r], 1);
      mbar_init(&pt_full[r], 128);
    }
    mbar_init(&acc_full, 1);
    mbar_init(&acc_empty, kComputeWarps * 32);
    mbar_init(&drain, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  volatile uint32_t* abort_v = &abort_flag;
  const int G = p.G;

  if (warp >= 8) {
   regs_decrease<kRegsOtherKV>();
   if (warp == kLoadWarp) {
    // ------------------------------------------------------------ TMA producer
    // The prep kernel's vectors are complete before the first load; then the dQ
    // kernel may be scheduled (its CTAs take the SMs this kernel's CTAs leave).
    ATTN_TR_DECL(0, 0, lane == 0);
    ATTN_TR(0, 0);  // CTA start
    griddep_wait();
    griddep_launch_dependents();
    uint32_t it = 0, n_ne = 0;  // ring loads issued; items with query tiles
    bool ok = true;
    for (int k = 0; k * static_cast<int>(gridDim.x) < p.n_items && ok; ++k) {
      const int x = item_of(k);
      if (x >= p.n_items) continue;
      const int j = x / nz, z = x % nz;
      const int i0 = first_qtile(p, j);
      const int nI = p.n_qt - i0;
      if (nI <= 0) continue;
      if (n_ne > 0) ok = warp_wait(&kv_empty, (n_ne - 1) & 1, abort_v, kTimeoutNs);
      if (!ok) break;
      ATTN_TR(1, x);  // the item's K and V loads issued
      mbar_arrive_expect_tx_elect(&kv_full, 2 * C::kTileBytes);
#pragma unroll
      for (int cb = 0; cb < D / 64; ++cb) {
        tma_load_3d_elect(k_s + cb * C::kColBlockBytes, &tk, &kv_full, cb * 64, j * BT, z);
        tma_load_3d_elect(v_s + cb * C::kColBlockBytes, &tv, &kv_full, cb * 64, j * BT, z);
      }
      ++n_ne;
      const int b = z / p.Hkv, kvh = z % p.Hkv;
      for (int s = 0; s < G * nI && ok; ++s, ++it) {
        const int h = kvh * G + s / nI, i = i0 + s % nI;
        const int bh = b * p.Hq + h;
        const uint32_t slot = it % kRing, use = it / kRing;
        if (use > 0) ok = warp_wait(&empty[slot], (use - 1) & 1, abort_v, kTimeoutNs);
        if (!ok) break;
        uint8_t* sl = ring + slot * C::kSlotBytes;
        mbar_arrive_expect_tx_elect(&full[slot], 2 * C::kTileBytes + 2 * C::kVecBytes);
#pragma unroll
        for (int cb = 0; cb < D / 64; ++cb) {
          tma_load_3d_elect(sl + cb * C::kColBlockBytes, &tq, &full[slot], cb * 64, i * BT, bh);
          tma_load_3d_elect(sl + C::kTileBytes + cb * C::kColBlockBytes, &tdo, &full[slot], cb * 64, i * BT, bh);
        }
        const int64_t voff = static_cast<int64_t>(bh) * p.Sq_pad + i * BT;
        bulk_load_1d_elect(sl + 2 * C::kTileBytes, p.nlse2 + voff, C::kVecBytes, &full[slot]);
        bulk_load_1d_elect(sl + 2 * C::kTileBytes + C::kVecBytes, p.ndelta + voff, C::kVecBytes, &full[slot]);
      }
    }
    if (!ok) {
      if (lane == 0) record_abort(abort_v, kSiteProducer);
      for (uint32_t u = (it > kRing ? it - kRing : 0); u < it; ++u)
        mbar_wait_bounded(&full[u % kRing], (u / kRing) & 1, abort_v, kDrainTimeoutNs);
      if (n_ne > 0) mbar_wait_bounded(&kv_full, (n_ne - 1) & 1, abort_v, kDrainTimeoutNs);
    }
    ATTN_TR_DONE();
   } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ tcgen05 issuer
    constexpr uint32_t idesc_s = idesc_bf16_f32(BT, BH2, false);  // M = 128 keys, N = 64 query rows
    constexpr uint32_t idesc_acc = idesc_bf16_f32(BT, D, true);   // M = 128 keys, N = D, B MN-major
    const uint32_t k_addr = smem_u32(k_s), v_addr = smem_u32(v_s), ring_addr = smem_u32(ring);
    // S^T_r = K Q_r^T and dP^T_r = V dO_r^T for half r of the query tile in ring slot `slot`
    // (K steps over D; a half starts 64 rows = kHalfBytes into each 64-column block)
    auto issue_s = [&](int r, uint32_t slot) {
      const uint32_t q_addr = opaque(ring_addr) + slot * C::kSlotBytes + r * kHalfBytes;
      const uint64_t kd = sdesc_sw128(k_addr, 16, 1024), vd = sdesc_sw128(v_addr, 16, 1024);
      const uint64_t qd = sdesc_sw128(q_addr, 16, 1024), dod = sdesc_sw128(q_addr + C::kTileBytes, 16, 1024);
      if constexpr (D == 128) {
        mma_bf16_ss_k8(tmem + 128 * r, kd, qd, idesc_s);
        mma_bf16_ss_k8(tmem + 128 * r + BH2, vd, dod, idesc_s, smem_u32(&st_full[r]));
      } else {
        mma_bf16_ss_k4(tmem + 128 * r, kd, qd, idesc_s);
        mma_bf16_ss_k4(tmem + 128 * r + BH2, vd, dod, idesc_s, smem_u32(&st_full[r]));
      }
    };
    // dV += P^T_r dO_r and dK += dS^T_r Q_r: A from TMEM (K = the half's 64 rows), B (dO, Q)
    // MN-major over those rows
    auto issue_acc = [&](int r, uint32_t slot, uint32_t acc, uint32_t bar0, uint32_t bar1) {
      const uint32_t q_addr = opaque(ring_addr) + slot * C::kSlotBytes + r * kHalfBytes;
      const uint64_t dob = sdesc_sw128(q_addr + C::kTileBytes, C::kColBlockBytes, 1024);
      const uint64_t qb = sdesc_sw128(q_addr, C::kColBlockBytes, 1024);
      mma_bf16_ts_k4(tmem + 2 * BT, tmem + 128 * r, dob, idesc_acc, acc);
      mma_bf16_ts_k4(tmem + 3 * BT, tmem + 128 * r + BH2, qb, idesc_acc, acc, bar0, bar1);
    };
    ATTN_TR_DECL(0, 1, lane == 0);
    uint32_t it = 0, g = 0, n_ne = 0;  // ring uses, steps (st/pt phases), items with query tiles
    bool ok = true;
    for (int k = 0; k * static_cast<int>(gridDim.x) < p.n_items && ok; ++k) {
      const int x = item_of(k);
      if (x >= p.n_items) continue;
      const int j = x / nz;
      const int nI = p.n_qt - first_qtile(p, j);
      if (nI <= 0) continue;
      const int T = G * nI;  // steps of the item
      ok = warp_wait(&kv_full, n_ne & 1, abort_v, kTimeoutNs);
      if (ok) ok = warp_wait(&full[it % kRing], (it / kRing) & 1, abort_v, kTimeoutNs);
      if (!ok) break;
      tc_fence_after();
      ATTN_TR(10, x);  // the item's first S-type products
      issue_s(0, it % kRing);
      issue_s(1, it % kRing);
      // K and V are read only by the S-type products: the next item's K and V may load
      // once the item's last ones have been issued and completed
      if (T == 1) mma_commit_elect(&kv_empty);
      for (int s = 0; s < T; ++s, ++it, ++g) {
        const uint32_t slot = it % kRing, next = (it + 1) % kRing;
        const bool more = s + 1 < T;
        ok = warp_wait(&pt_full[0], g & 1, abort_v, kTimeoutNs);
        if (ok && s == 0 && n_ne > 0) ok = warp_wait(&acc_empty, (n_ne - 1) & 1, abort_v, kTimeoutNs);
        if (!ok) break;
        tc_fence_after();
        issue_acc(0, slot, s > 0 ? 1u : 0u, kNoBar, kNoBar);
        ATTN_TR(11, s);  // half 0's dV and dK products of step s
        if (more) {
          ok = warp_wait(&full[next], ((it + 1) / kRing) & 1, abort_v, kTimeoutNs);
          if (!ok) break;
          tc_fence_after();
          issue_s(0, next);  // region 0 is free once the MMAs just issued have read it
        }
        ok = warp_wait(&pt_full[1], g & 1, abort_v, kTimeoutNs);
        if (!ok) break;
        tc_fence_after();
        // half 1's products are the slot's last readers; the item's last one completes dV and dK
        issue_acc(1, slot, 1u, smem_u32(&empty[slot]), more ? kNoBar : smem_u32(&acc_full));
        if (more) issue_s(1, next);
        if (s + 2 == T) mma_commit_elect(&kv_empty);  // that was the item's last S-type pair
      }
      if (!ok) break;
      ++n_ne;
    }
    if (!ok && lane == 0) record_abort(abort_v, kSiteIssuer);
    mma_commit_elect(&drain);
    warp_wait(&drain, 0, abort_v, ok ? kTimeoutNs : kDrainTimeoutNs);
    ATTN_TR(13, 0);  // every MMA of the CTA completed
    ATTN_TR_DONE();
   }
  } else {
    // ------------------------------------------------------------ compute (one thread per key)
    // Warpgroup r takes half r (query rows 64 r .. 64 r + 63) of every step: the thread of
    // key kk reads its lane of S^T_r and dP^T_r (64 columns each) and writes P^T_r and
    // dS^T_r over their first 32 columns, its own lane only.  At the end of an item
    // warpgroup 0 writes dV, warpgroup 1 scale * dK.
    regs_increase<kRegsComputeKV>();
    const int r = warp / 4, quarter = warp % 4;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t st_t = tmem + lane_off + 128 * r, dpt_t = st_t + BH2;
    const uint32_t acc_t = tmem + lane_off + (r == 0 ? 2 * BT : 3 * BT);
    const int kk = quarter * 32 + lane;
    ATTN_TR_DECL(0, 2 + r, quarter == 0 && lane == 0);
    uint32_t it = 0, g = 0, n_ne = 0;
    bool ok = true;
    for (int k = 0; k * static_cast<int>(gridDim.x) < p.n_items && ok; ++k) {
      const int x = item_of(k);
      if (x >= p.n_items) continue;
      const int j = x / nz;
      const int i0 = first_qtile(p, j);
      const int nI = p.n_qt - i0;
      const int key = j * BT + kk;
      const bool key_live = key < p.Sk;
      // this key's dV (warpgroup 0) or dK (warpgroup 1) row
      auto grad_row = [&]() { return (r == 0 ? p.dv : p.dk) + (static_cast<int64_t>(x % nz) * p.Sk + key) * D; };
      if (nI <= 0) {  // no query row sees this key tile: zero gradients
        if (key_live) {
          uint4* a4 = reinterpret_cast<uint4*>(grad_row());
#pragma unroll
          for (int v4 = 0; v4 < D / 8; ++v4) a4[v4] = make_uint4(0u, 0u, 0u, 0u);
        }
        continue;
      }
      for (int s = 0; s < G * nI; ++s, ++it, ++g) {
        const int i = i0 + s % nI;
        const uint8_t* sl = ring + (it % kRing) * C::kSlotBytes;
        const float4* nl4 = reinterpret_cast<const float4*>(sl + 2 * C::kTileBytes) + (BH2 / 4) * r;
        const float4* nd4 = reinterpret_cast<const float4*>(sl + 2 * C::kTileBytes + C::kVecBytes) + (BH2 / 4) * r;
        // the slot's vectors have landed (this warp observes their copy itself), then S^T_r and dP^T_r
        ok = warp_wait(&full[it % kRing], (it / kRing) & 1, abort_v, kTimeoutNs);
        if (ok) ok = warp_wait(&st_full[r], g & 1, abort_v, kTimeoutNs);
        if (!ok) break;
        ATTN_TR(20, s);  // S^T_r and dP^T_r of step s ready
        tc_fence_after();
        uint32_t sv[64], dpv[64];
        tmem_ld2x64_wait(st_t, dpt_t, sv, dpv);
        // masked elements (keys past Sk, keys above the diagonal of a straddling tile) get
        // S = -inf, hence P = 0 (c > 0)
        const bool diag_tile = p.causal && (j * BT + BT - 1 > i * BT + p.diag);
        if (__any_sync(0xffffffffu, diag_tile || !key_live)) {
          const int first_ok = key_live ? (diag_tile ? key - p.diag - i * BT - BH2 * r : 0) : BH2;
#pragma unroll
          for (int e = 0; e < 64; ++e) sv[e] = e >= first_ok ? sv[e] : __float_as_uint(-INFINITY);
        }
        // P = exp2(S c - LSE log2 e) and dS = P (dP - D), two rows per packed operation
        const uint64_t c2 = f2_pack(p.c, p.c);
        uint32_t pk[32], dsk[32];
#pragma unroll
        for (int r4 = 0; r4 < 16; ++r4) {
          const float4 l4 = nl4[r4], d4 = nd4[r4];
          const float lv[4] = {l4.x, l4.y, l4.z, l4.w}, dl[4] = {d4.x, d4.y, d4.z, d4.w};
          float pp[4], dd[4];
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            const int e = 4 * r4 + h;
            pp[h] = ex2_approx(fmaf(__uint_as_float(sv[e]), p.c, lv[h]));
          }
          float y0, y1, y2, y3;
          f2_unpack(fmul2(f2_pack(pp[0], pp[1]), fadd2(f2_pack(__uint_as_float(dpv[4 * r4]), __uint_as_float(dpv[4 * r4 + 1])), f2_pack(dl[0], dl[1]))), y0, y1);
          f2_unpack(fmul2(f2_pack(pp[2], pp[3]), fadd2(f2_pack(__uint_as_float(dpv[4 * r4 + 2]), __uint_as_float(dpv[4 * r4 + 3])), f2_pack(dl[2], dl[3]))), y2, y3);
          dd[0] = y0; dd[1] = y1; dd[2] = y2; dd[3] = y3;
          pk[2 * r4] = pack_bf16x2(pp[0], pp[1]);
          pk[2 * r4 + 1] = pack_bf16x2(pp[2], pp[3]);
          dsk[2 * r4] = pack_bf16x2(dd[0], dd[1]);
          dsk[2 * r4 + 1] = pack_bf16x2(dd[2], dd[3]);
        }
        tmem_st32(st_t, pk);
        tmem_st32(dpt_t, dsk);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&pt_full[r]);
        ATTN_TR(21, s);  // P^T_r and dS^T_r handed to the MMA
      }
      if (!ok) break;
      // epilogue: dV (warpgroup 0) or scale * dK (warpgroup 1) of this key, bf16, once the
      // item's MMAs are done
      ok = warp_wait(&acc_full, n_ne & 1, abort_v, kTimeoutNs);
      if (!ok) break;
      ATTN_TR(23, x);  // the item's dV and dK complete: epilogue starts
      ++n_ne;
      tc_fence_after();
      const float mul = r == 0 ? 1.0f : p.scale;
      // the warp's 32 keys' rows, 64 bytes (32 columns) at a time
      uint8_t* wbase = reinterpret_cast<uint8_t*>(grad_row() - lane * D);
      const int live_keys = p.Sk - (j * BT + quarter * 32);
#pragma unroll
      for (int cb = 0; cb < D / 32; ++cb) {
        uint32_t a[32], w[16];
        tmem_ld32_wait(acc_t + 32 * cb, a);
#pragma unroll
        for (int e = 0; e < 16; ++e)
          w[e] = pack_bf16x2(__uint_as_float(a[2 * e]) * mul, __uint_as_float(a[2 * e + 1]) * mul);
        store_warp_rows<4>(w, wbase + 64 * cb, 2 * D, live_keys, lane);
      }
      tc_fence_before();
      mbar_arrive(&acc_empty);  // dV and dK may be overwritten by the next item
      ATTN_TR(24, x);  // epilogue done
    }
    if (!ok && lane == 0) record_abort(abort_v, kSiteCompute);
    ATTN_TR_DONE();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Key tiles query tile i visits: [0, n).
__device__ __forceinline__ int key_tiles(const BParams& p, int i) {
  if (!p.causal) return p.n_kt;
  const int last_row = min(i * BT + BT, p.Sq) - 1;
  const int kv_end = min(p.Sk, last_row + p.diag + 1);
  return kv_end > 0 ? (kv_end + BT - 1) / BT : 0;
}

// ---------------------------------------------------------------------------- dQ
// Work item x: query tile i = n_qt - 1 - x / (B*Hq) (heaviest first under a causal
// mask), slice bh = x % (B*Hq).  A step is one 128-key tile.  S = Q K^T of a step goes
// to one of two TMEM regions (steps alternate: [0,128) and [128,256)), dP = dO V^T to
// [256,384), dQ accumulates at [384, 384 + D) (lane = query row); both products are 128
// wide (a 64-wide product costs half again as many tensor cycles per FLOP).  Warpgroup r
// takes keys 64 r .. 64 r + 63 of every step and writes their dS (bf16 pairs) over its
// own S columns [64 r, 64 r + 32) of the step's region.  The next step's S and dP go in
// as soon as both warpgroups have read this step's dP, so the tensor cores compute them
// while the warpgroups work; K streams through a three-slot ring (it is read again by
// dQ += dS K) and V through a two-slot one.  Each warpgroup's dS-ready barrier is
// doubled by step parity so it can never get two phases ahead of the issuer.
template <int D>
struct QCfg {
  static constexpr int kTileBytes = BT * D * 2;
  static constexpr int kKRing = 3, kVRing = 2;
  static constexpr int kSmemBytes = (2 + kKRing + kVRing) * kTileBytes + 1024;  // Q, dO, K ring, V ring
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                       const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                       const BParams p) {
  using C = QCfg<D>;
  using BC = BCfg<D>;
  constexpr int KR = C::kKRing, VR = C::kVRing;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_1024(smem_raw);
  uint8_t* q_s = smem;
  uint8_t* do_s = smem + C::kTileBytes;
  uint8_t* k_ring = smem + 2 * C::kTileBytes;
  uint8_t* v_ring = k_ring + KR * C::kTileBytes;
  __shared__ uint64_t qd_full, qd_empty, kfull[KR], kempty[KR], vfull[VR], vempty[VR], st_full, dp_free,
      ds_full[2][2], acc_full, acc_empty, drain;
  __shared__ uint32_t tmem_slot, abort_flag;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    mbar_init(&qd_full, 1);
    mbar_init(&qd_empty, 1);
    for (int s = 0; s < KR; ++s) {
      mbar_init(&kfull[s], 1);
      mbar_init(&kempty[s], 1);
    }
    for (int s = 0; s < VR; ++s) {
      mbar_init(&vfull[s], 1);
      mbar_init(&vempty[s], 1);
    }
    mbar_init(&st_full, 1);
    mbar_init(&dp_free, kComputeWarps * 32);
    for (int r = 0; r < 2; ++r) {
      mbar_init(&ds_full[r][0], 128);
      mbar_init(&ds_full[r][1], 128);
    }
    mbar_init(&acc_full, 1);
    mbar_init(&acc_empty, kComputeWarps * 32);
    mbar_init(&drain, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  volatile uint32_t* abort_v = &abort_flag;

  if (warp >= 8) {
   regs_decrease<kRegsOther>();
   if (warp == kLoadWarp) {
    // ------------------------------------------------------------ TMA producer
    ATTN_TR_DECL(1, 0, lane == 0);
    ATTN_TR(0, 0);  // CTA start
    uint32_t kl = 0, vl = 0, n_ne = 0;  // K and V tiles loaded; items with key tiles
    bool ok = true;
    for (int k = 0; k * static_cast<int>(gridDim.x) < p.n_items && ok; ++k) {
      const int x = item_of(k);
      if (x >= p.n_items) continue;
      const int i = p.n_qt - 1 - x / p.BH, bh = x % p.BH;
      const int n = key_tiles(p, i);
      if (n <= 0) continue;
      if (n_ne > 0) ok = warp_wait(&qd_empty, (n_ne - 1) & 1, abort_v, kTimeoutNs);
      if (!ok) break;
      ATTN_TR(1, x);  // the item's Q and dO loads issued
      mbar_arrive_expect_tx_elect(&qd_full, 2 * C::kTileBytes);
#pragma unroll
      for (int cb = 0; cb < D / 64; ++cb) {
        tma_load_3d_elect(q_s + cb * BC::kColBlockBytes, &tq, &qd_full, cb * 64, i * BT, bh);
        tma_load_3d_elect(do_s + cb * BC::kColBlockBytes, &tdo, &qd_full, cb * 64, i * BT, bh);
      }
      ++n_ne;
      const int kvz = (bh / p.Hq) * p.Hkv + (bh % p.Hq) / p.G;
      for (int j = 0; j < n && ok; ++j, ++kl, ++vl) {
        const uint32_t ks = kl % KR, vs = vl % VR;
        if (kl >= KR) ok = warp_wait(&kempty[ks], (kl / KR - 1) & 1, abort_v, kTimeoutNs);
        if (!ok) break;
        mbar_arrive_expect_tx_elect(&kfull[ks], C::kTileBytes);
#pragma unroll
        for (int cb = 0; cb < D / 64; ++cb)
          tma_load_3d_elect(k_ring + ks * C::kTileBytes + cb * BC::kColBlockBytes, &tk, &kfull[ks], cb * 64, j * BT,
                            kvz);
        if (vl >= VR) ok = warp_wait(&vempty[vs], (vl / VR - 1) & 1, abort_v, kTimeoutNs);
        if (!ok) {
          ++kl;  // the K tile above is in flight
          break;
        }
        mbar_arrive_expect_tx_elect(&vfull[vs], C::kTileBytes);
#pragma unroll
        for (int cb = 0; cb < D / 64; ++cb)
          tma_load_3d_elect(v_ring + vs * C::kTileBytes + cb * BC::kColBlockBytes, &tv, &vfull[vs], cb * 64, j * BT,
                            kvz);
      }
    }
    if (!ok) {
      if (lane == 0) record_abort(abort_v, kSiteProducer);
      for (uint32_t u = (kl > KR ? kl - KR : 0); u < kl; ++u)
        mbar_wait_bounded(&kfull[u % KR], (u / KR) & 1, abort_v, kDrainTimeoutNs);
      for (uint32_t u = (vl > VR ? vl - VR : 0); u < vl; ++u)
        mbar_wait_bounded(&vfull[u % VR], (u / VR) & 1, abort_v, kDrainTimeoutNs);
      if (n_ne > 0) mbar_wait_bounded(&qd_full, (n_ne - 1) & 1, abort_v, kDrainTimeoutNs);
    }
    ATTN_TR_DONE();
   } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ tcgen05 issuer
    ATTN_TR_DECL(1, 1, lane == 0);
    constexpr uint32_t idesc_s = idesc_bf16_f32(BT, BT, false);  // M = 128 rows, N = 128 keys
    constexpr uint32_t idesc_acc = idesc_bf16_f32(BT, D, true);  // M = 128 rows, N = D, B MN-major
    constexpr uint32_t kDp = 2 * BT, kDq = 3 * BT;               // TMEM columns of dP and dQ
    const uint32_t q_addr = smem_u32(q_s), do_addr = smem_u32(do_s);
    const uint32_t k_addr = smem_u32(k_ring), v_addr = smem_u32(v_ring);
    // S = Q K^T into TMEM region `reg`
    auto issue_s = [&](uint32_t reg, uint32_t ks) {
      const uint64_t qd = sdesc_sw128(q_addr, 16, 1024);
      const uint64_t kd = sdesc_sw128(opaque(k_addr) + ks * C::kTileBytes, 16, 1024);
      if constexpr (D == 128)
        mma_bf16_ss_k8(tmem + reg, qd, kd, idesc_s);
      else
        mma_bf16_ss_k4(tmem + reg, qd, kd, idesc_s);
    };
    // dP = dO V^T; the step's S and dP are then ready, and V is free
    auto issue_dp = [&](uint32_t vs) {
      const uint64_t dod = sdesc_sw128(do_addr, 16, 1024);
      const uint64_t vd = sdesc_sw128(opaque(v_addr) + vs * C::kTileBytes, 16, 1024);
      if constexpr (D == 128)
        mma_bf16_ss_k8(tmem + kDp, dod, vd, idesc_s, smem_u32(&st_full), smem_u32(&vempty[vs]));
      else
        mma_bf16_ss_k4(tmem + kDp, dod, vd, idesc_s, smem_u32(&st_full), smem_u32(&vempty[vs]));
    };
    // dQ += dS K for step gg (dS in region gg & 1, K in slot ks), one 64-key half per
    // warpgroup as its dS arrives; the item's first step overwrites dQ once the previous
    // item's epilogue has read it, its last commits acc_full; K is free afterwards
    auto issue_acc = [&](uint32_t gg, uint32_t ks, bool first, bool last, uint32_t tt) -> bool {
      const uint32_t reg = tmem + BT * (gg & 1), ka = opaque(k_addr) + ks * C::kTileBytes;
      bool w = warp_wait(&ds_full[0][gg & 1], (gg >> 1) & 1, abort_v, kTimeoutNs);
      if (w && first && tt > 0) w = warp_wait(&acc_empty, (tt - 1) & 1, abort_v, kTimeoutNs);
      if (!w) return false;
      tc_fence_after();
      mma_bf16_ts_k4(tmem + kDq, reg, sdesc_sw128(ka, BC::kColBlockBytes, 1024), idesc_acc, first ? 0u : 1u);
      ATTN_TR(11, (first ? 0u : 1u) | (last ? 2u : 0u));  // half 0's dQ += dS K (arg: item's first, last)
      w = warp_wait(&ds_full[1][gg & 1], (gg >> 1) & 1, abort_v, kTimeoutNs);
      if (!w) return false;
      tc_fence_after();
      mma_bf16_ts_k4(tmem + kDq, reg + BH2, sdesc_sw128(ka + kHalfBytes, BC::kColBlockBytes, 1024), idesc_acc, 1u,
                     smem_u32(&kempty[ks]), last ? smem_u32(&acc_full) : kNoBar);
      return true;
    };
    // Order on the tensor pipe: S(g) dP(g) dQ+=(g-1) S(g+1) dP(g+1) dQ+=(g) ..., across items too.
    // S(g) overwrites step g-2's region, whose S was read before dP(g-1) went in and whose dS
    // was consumed by the products issued before it, so it is issued without waiting for the
    // warpgroups; only dP(g) waits for them to have read dP(g-1).
    uint32_t g = 0, t = 0;    // steps (= K and V tiles), items with key tiles
    uint32_t pk = 0, pt = 0;  // the step whose dQ += dS K is pending: K slot, item
    int pj = -1, pn = 0;      // ... and its index within the item, the item's steps
    bool ok = true;
    for (int k = 0; k * static_cast<int>(gridDim.x) < p.n_items && ok; ++k) {
      const int x = item_of(k);
      if (x >= p.n_items) continue;
      const int n = key_tiles(p, p.n_qt - 1 - x / p.BH);
      if (n <= 0) continue;
      ok = warp_wait(&qd_full, t & 1, abort_v, kTimeoutNs);
      for (int j = 0; j < n && ok; ++j, ++g) {
        const uint32_t ks = g % KR, vs = g % VR;
        ok = warp_wait(&kfull[ks], (g / KR) & 1, abort_v, kTimeoutNs);
        if (!ok) break;
        tc_fence_after();
        if (j == 0) ATTN_TR(10, x);  // the item's first S product
        issue_s(BT * (g & 1), ks);
        if (g > 0) ok = warp_wait(&dp_free, (g - 1) & 1, abort_v, kTimeoutNs);  // dP(g-1) read by all
        if (ok) ok = warp_wait(&vfull[vs], (g / VR) & 1, abort_v, kTimeoutNs);
        if (!ok) break;
        tc_fence_after();
        issue_dp(vs);
        if (j + 1 == n) mma_commit_elect(&qd_empty);  // Q and dO are read only by S and dP
        if (pj >= 0) ok = issue_acc(g - 1, pk, pj == 0, pj + 1 == pn, pt);
        pk = ks;
        pj = j;
        pn = n;
        pt = t;
      }
      if (!ok) break;
      ++t;
    }
    if (ok && pj >= 0) ok = issue_acc(g - 1, pk, pj == 0, pj + 1 == pn, pt);
    if (!ok && lane == 0) record_abort(abort_v, kSiteIssuer);
    mma_commit_elect(&drain);
    warp_wait(&drain, 0, abort_v, ok ? kTimeoutNs : kDrainTimeoutNs);
    ATTN_TR(13, 0);  // every MMA of the CTA completed
    ATTN_TR_DONE();
   }
  } else {
    // ------------------------------------------------------------ compute (one thread per query row)
    // Warpgroup r takes keys 64 r .. 64 r + 63 of every key tile; at the end of an item it
    // writes columns r * D/2 .. of the row's dQ.
    regs_increase<kRegsCompute>();
    const int r = warp / 4, quarter = warp % 4;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t dp_t = tmem + lane_off + 2 * BT + BH2 * r, dq_t = tmem + lane_off + 3 * BT;
    ATTN_TR_DECL(1, 2 + r, quarter == 0 && lane == 0);
    uint32_t g = 0, t = 0;
    bool ok = true;
    for (int k = 0; k * static_cast<int>(gridDim.x) < p.n_items && ok; ++k) {
      const int x = item_of(k);
      if (x >= p.n_items) continue;
      const int i = p.n_qt - 1 - x / p.BH, bh = x % p.BH;
      const int n = key_tiles(p, i);
      const int row = i * BT + quarter * 32 + lane;
      const bool live = row < p.Sq;
      __nv_bfloat16* dqrow = p.dq + (static_cast<int64_t>(bh) * p.Sq + row) * D + r * (D / 2);
      if (n <= 0) {  // no key is visible to any row of this tile: zero gradient
        if (live) {
          uint4* a4 = reinterpret_cast<uint4*>(dqrow);
#pragma unroll
          for (int v4 = 0; v4 < D / 16; ++v4) a4[v4] = make_uint4(0u, 0u, 0u, 0u);
        }
        continue;
      }
      const float nl = p.nlse2[static_cast<int64_t>(bh) * p.Sq_pad + row];
      const float nd = p.ndelta[static_cast<int64_t>(bh) * p.Sq_pad + row];
      const uint64_t c2 = f2_pack(p.c, p.c), nl2 = f2_pack(nl, nl), nd2 = f2_pack(nd, nd);
      const int lim = p.causal ? min(p.Sk - 1, row + p.diag) : p.Sk - 1;  // last visible key
      for (int j = 0; j < n; ++j, ++g) {
        ok = warp_wait(&st_full, g & 1, abort_v, kTimeoutNs);
        if (!ok) break;
        ATTN_TR(20, j);  // S and dP of key tile j ready
        tc_fence_after();
        const uint32_t s_t = tmem + lane_off + BT * (g & 1) + BH2 * r;
        uint32_t sv[64], dpv[64];
        tmem_ld2x64_wait(s_t, dp_t, sv, dpv);
        tc_fence_before();
        mbar_arrive(&dp_free);  // the next step's S and dP may go in
        // keys past kmax (above the diagonal, or past Sk) get S = -inf, hence P = 0 (c > 0)
        const int kmax = lim - j * BT - BH2 * r;
        if (__any_sync(0xffffffffu, kmax < BH2 - 1)) {
#pragma unroll
          for (int e = 0; e < 64; ++e) sv[e] = e <= kmax ? sv[e] : __float_as_uint(-INFINITY);
        }
        // dS = P (dP - D) with P = exp2(S c - LSE log2 e), two keys per packed operation
        uint32_t dsk[32];
#pragma unroll
        for (int e2 = 0; e2 < 32; ++e2) {
          float x0, x1, y0, y1;
          f2_unpack(ffma2(f2_pack(__uint_as_float(sv[2 * e2]), __uint_as_float(sv[2 * e2 + 1])), c2, nl2), x0, x1);
          const uint64_t pp = f2_pack(ex2_approx(x0), ex2_approx(x1));
          const uint64_t dp = fadd2(f2_pack(__uint_as_float(dpv[2 * e2]), __uint_as_float(dpv[2 * e2 + 1])), nd2);
          f2_unpack(fmul2(pp, dp), y0, y1);
          dsk[e2] = pack_bf16x2(y0, y1);
        }
        tmem_st32(s_t, dsk);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&ds_full[r][g & 1]);
        ATTN_TR(21, j);  // dS of this warpgroup's keys handed to the MMA
      }
      if (!ok) break;
      ok = warp_wait(&acc_full, t & 1, abort_v, kTimeoutNs);
      if (!ok) break;
      ATTN_TR(23, x);  // the item's dQ complete: epilogue starts
      ++t;
      tc_fence_after();
      // the warp's 32 rows, this warpgroup's D/2 columns (D bytes) of each
      {
        constexpr int CH = D / 16;
        uint32_t w[4 * CH];
#pragma unroll
        for (int cb = 0; cb < D / 64; ++cb) {
          uint32_t a[32];
          tmem_ld32_wait(dq_t + r * (D / 2) + 32 * cb, a);
#pragma unroll
          for (int e = 0; e < 16; ++e)
            w[16 * cb + e] = pack_bf16x2(__uint_as_float(a[2 * e]) * p.scale, __uint_as_float(a[2 * e + 1]) * p.scale);
        }
        store_warp_rows<CH>(w, reinterpret_cast<uint8_t*>(dqrow - lane * D), 2 * D, p.Sq - (i * BT + quarter * 32),
                            lane);
      }
      tc_fence_before();
      mbar_arrive(&acc_empty);
      ATTN_TR(24, x);  // epilogue done
    }
    if (!ok && lane == 0) record_abort(abort_v, kSiteCompute);
    ATTN_TR_DONE();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  // this grid may run beside the tail of the dK/dV kernel (it reads only the prep
  // kernel's vectors, complete before the dK/dV kernel let it start); it completes
  // after that kernel, so work later in the stream sees all three gradients
  if (threadIdx.x == 0) griddep_wait();
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
std::mutex g_dev_mutex;
int g_dev_state[kMaxDevices];  // 0 unknown, 1 ready, -1 unsupported
int g_dev_sms[kMaxDevices];

int prepare_device(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  if (g_dev_state[dev] == 1) return ATTN_OK;
  if (g_dev_state[dev] == -1) return ATTN_ERR_UNSUPPORTED_DEVICE;
  int major = 0, minor = 0, sms = 0;
  cudaError_t e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (major != 10 || minor != 3) {
    g_dev_state[dev] = -1;
    return ATTN_ERR_UNSUPPORTED_DEVICE;
  }
  g_dev_sms[dev] = sms;
  const void* fns[] = {reinterpret_cast<const void*>(attn_bwd_dkdv_kernel<128>),
                       reinterpret_cast<const void*>(attn_bwd_dq_kernel<128>),
                       reinterpret_cast<const void*>(attn_bwd_dkdv_kernel<64>),
                       reinterpret_cast<const void*>(attn_bwd_dq_kernel<64>)};
  const int bytes[] = {BCfg<128>::kSmemBytes, QCfg<128>::kSmemBytes, BCfg<64>::kSmemBytes, QCfg<64>::kSmemBytes};
  for (int f = 0; f < 4 && e == cudaSuccess; ++f)
    e = cudaFuncSetAttribute(fns[f], cudaFuncAttributeMaxDynamicSharedMemorySize, bytes[f]);
  if (e != cudaSuccess) return cuda_fail(e);
  if (!attn_host::encode_tiled_fn()) return ATTN_ERR_TENSOR_MAP;
  g_dev_state[dev] = 1;
  return ATTN_OK;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  if (!a || !b || na == 0 || nb == 0) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + nb && b0 < a0 + na;
}

bool misaligned(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) != 0; }

int64_t padded_rows(int Sq) { return (static_cast<int64_t>(Sq) + BT - 1) / BT * BT; }

template <int D>
int launch_all(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
               BParams prm, const __nv_bfloat16* o, const __nv_bfloat16* dout, const float* lse, float* lse2,
               float* delta, int sms, cudaStream_t stream) {
  const int64_t prep_rows = static_cast<int64_t>(prm.BH) * prm.Sq_pad;
  const int64_t prep_warps = (prep_rows + 32 / (D / 8) - 1) / (32 / (D / 8));
  attn_bwd_prep_kernel<D><<<static_cast<unsigned>((prep_warps + 7) / 8), 256, 0, stream>>>(
      o, dout, lse, lse2, delta, prm.BH, prm.Sq, prm.Sq_pad);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e);
  // the dK/dV and dQ kernels are launched with programmatic stream serialisation: each
  // may be scheduled before the previous kernel has finished (see griddep_* in ptx.cuh)
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = BCfg<D>::kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  BParams a = prm;
  a.n_items = prm.n_kt * prm.BZ;
  cfg.gridDim = dim3(a.n_items < sms ? a.n_items : sms);
  e = cudaLaunchKernelEx(&cfg, attn_bwd_dkdv_kernel<D>, tq, tk, tv, tdo, a);
  if (e != cudaSuccess) return cuda_fail(e);
  BParams b = prm;
  b.n_items = prm.n_qt * prm.BH;
  cfg.gridDim = dim3(b.n_items < sms ? b.n_items : sms);
  cfg.dynamicSmemBytes = QCfg<D>::kSmemBytes;
  e = cudaLaunchKernelEx(&cfg, attn_bwd_dq_kernel<D>, tq, tk, tv, tdo, b);
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}

}  // namespace

extern "C" {

size_t attn_bwd_workspace_size(int B, int Hq, int Sq) {
  if (B < 0 || Hq < 1 || Sq < 0) return 0;
  const size_t one = static_cast<size_t>(B) * Hq * padded_rows(Sq) * 4;
  return 2 * ((one + 255) & ~static_cast<size_t>(255));
}

int attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
             void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Sq, int Sk, int D, int causal, float scale,
             void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  // ---- argument checks (host only, before any CUDA call)
  if (B < 0 || Sq < 0 || Sk < 0 || Hq < 1 || Hkv < 1) return ATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return ATTN_ERR_INVALID_ARG;
  if (Hq % Hkv != 0 || causal < 0 || causal > 2 || !(std::isfinite(scale) && scale > 0.0f)) return ATTN_ERR_INVALID_ARG;
  if (static_cast<int64_t>(B) * Hq > INT32_MAX / 2 || padded_rows(Sq) > INT32_MAX / 2) return ATTN_ERR_INVALID_ARG;
  if (B == 0) return ATTN_OK;
  const size_t qb = static_cast<size_t>(B) * Hq * Sq * D * 2, kb = static_cast<size_t>(B) * Hkv * Sk * D * 2;
  const size_t lb = static_cast<size_t>(B) * Hq * Sq * 4;
  const size_t wb = attn_bwd_workspace_size(B, Hq, Sq);
  if (Sq > 0 && (!q || !o || !lse || !dout || !dq)) return ATTN_ERR_NULL_PTR;
  if (Sk > 0 && (!k || !v || !dk || !dv)) return ATTN_ERR_NULL_PTR;
  if (Sq > 0 && Sk > 0 && !workspace) return ATTN_ERR_NULL_PTR;
  const void* al[] = {q, k, v, o, lse, dout, dq, dk, dv, workspace};
  for (const void* ptr : al)
    if (ptr && misaligned(ptr)) return ATTN_ERR_MISALIGNED;
  if (Sq > 0 && Sk > 0 && workspace_bytes < wb) return ATTN_ERR_INVALID_ARG;
  // outputs (and the workspace) must not overlap each other or any input
  const void* outs[] = {dq, dk, dv, workspace};
  const size_t out_n[] = {qb, kb, kb, wb};
  const void* ins[] = {q, k, v, o, lse, dout};
  const size_t in_n[] = {qb, kb, kb, qb, lb, qb};
  for (int a = 0; a < 4; ++a) {
    for (int b2 = 0; b2 < 6; ++b2)
      if (overlaps(outs[a], out_n[a], ins[b2], in_n[b2])) return ATTN_ERR_INVALID_ARG;
    for (int b2 = a + 1; b2 < 4; ++b2)
      if (overlaps(outs[a], out_n[a], outs[b2], out_n[b2])) return ATTN_ERR_INVALID_ARG;
  }

  // ---- device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  const int st = prepare_device(dev);
  if (st != ATTN_OK) return st;
  if (Sq == 0 || Sk == 0) {  // no (row, key) pair: the gradients that exist are zero
    if (Sk > 0) {
      if ((e = cudaMemsetAsync(dk, 0, kb, stream)) != cudaSuccess) return cuda_fail(e);
      if ((e = cudaMemsetAsync(dv, 0, kb, stream)) != cudaSuccess) return cuda_fail(e);
    }
    if (Sq > 0 && (e = cudaMemsetAsync(dq, 0, qb, stream)) != cudaSuccess) return cuda_fail(e);
    return ATTN_OK;
  }

  CUtensorMap tq, tk, tv, tdo;
  if (!attn_host::encode_bf16_rows(&tq, q, D, Sq, static_cast<uint64_t>(B) * Hq, BT) ||
      !attn_host::encode_bf16_rows(&tdo, dout, D, Sq, static_cast<uint64_t>(B) * Hq, BT) ||
      !attn_host::encode_bf16_rows(&tk, k, D, Sk, static_cast<uint64_t>(B) * Hkv, BT) ||
      !attn_host::encode_bf16_rows(&tv, v, D, Sk, static_cast<uint64_t>(B) * Hkv, BT))
    return ATTN_ERR_TENSOR_MAP;

  BParams prm;
  prm.dq = static_cast<__nv_bfloat16*>(dq);
  prm.dk = static_cast<__nv_bfloat16*>(dk);
  prm.dv = static_cast<__nv_bfloat16*>(dv);
  const size_t one = wb / 2;
  float* lse2 = static_cast<float*>(workspace);  // stored negated, as the kernels use them
  float* delta = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + one);
  prm.nlse2 = lse2;
  prm.ndelta = delta;
  prm.Hq = Hq;
  prm.Hkv = Hkv;
  prm.G = Hq / Hkv;
  prm.Sq = Sq;
  prm.Sk = Sk;
  prm.Sq_pad = static_cast<int>(padded_rows(Sq));
  prm.causal = causal != 0;
  prm.diag = causal == 1 ? Sk - Sq : 0;
  prm.n_qt = (Sq + BT - 1) / BT;
  prm.n_kt = (Sk + BT - 1) / BT;
  prm.BZ = B * Hkv;
  prm.BH = B * Hq;
  prm.n_items = 0;
  prm.c = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634074);
  prm.scale = scale;
  const auto* ob = static_cast<const __nv_bfloat16*>(o);
  const auto* gb = static_cast<const __nv_bfloat16*>(dout);
  return D == 128 ? launch_all<128>(tq, tk, tv, tdo, prm, ob, gb, lse, lse2, delta, g_dev_sms[dev], stream)
                  : launch_all<64>(tq, tk, tv, tdo, prm, ob, gb, lse, lse2, delta, g_dev_sms[dev], stream);
}

const char* attn_bwd_strerror(int status) {
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

#ifdef ATTN_TRACE
int attn_bwd_trace_read(void* dst, size_t dst_bytes, int* kernels, int* ctas, int* roles, int* events) {
  if (kernels) *kernels = kTraceKernels;
  if (ctas) *ctas = kTraceCtas;
  if (roles) *roles = kTraceRoles;
  if (events) *events = kTraceEvents;
  const size_t n_bytes = sizeof(unsigned int) * kTraceKernels * kTraceCtas * kTraceRoles;
  const size_t r_bytes = sizeof(TraceRec) * static_cast<size_t>(kTraceKernels) * kTraceCtas * kTraceRoles * kTraceEvents;
  if (!dst) return ATTN_ERR_NULL_PTR;
  if (dst_bytes < n_bytes + r_bytes) return ATTN_ERR_INVALID_ARG;
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(dst, g_btrace_n, n_bytes);
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(static_cast<uint8_t*>(dst) + n_bytes, g_btrace, r_bytes);
  static const unsigned int zeros[kTraceKernels * kTraceCtas * kTraceRoles] = {};  // later launches start empty
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_btrace_n, zeros, n_bytes);
  return e == cudaSuccess ? ATTN_OK : cuda_fail(e);
}
#endif

int attn_bwd_debug_status(cudaStream_t stream, int* site) {
  if (site) *site = 0;
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e);
  int value = 0;
  e = cudaMemcpyFromSymbol(&value, g_bwd_status, sizeof(int));
  if (e != cudaSuccess) return cuda_fail(e);
  if (value != 0) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_bwd_status, &zero, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e);
  }
  if (site) *site = value;
  return value == 0 ? ATTN_OK : ATTN_ERR_DEVICE_TIMEOUT;
}

}  // extern "C"
