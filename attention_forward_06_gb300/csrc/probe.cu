// probe.cu -- primitive kernels that check, one building block at a time, the
// hand-encoded pieces the attention kernel is made of:
//   * a TMA tile load with 128-byte swizzle and zero fill past the last row;
//   * S = Q K^T with both operands K-major in shared memory (SS form), the
//     accumulator read back from tensor memory with tcgen05.ld;
//   * O = P V with P written into tensor memory by tcgen05.st (TS form) and V
//     MN-major in shared memory;
// and two rate probes: the dense bf16 tcgen05 MMA rate per SM and the ex2.approx
// rate per SM, behind the peak and the softmax bound the benchmark and the
// kernel's design use.
// Each runs as a single CTA of 128 threads on one 128-row tile; the tests
// compare the results with CPU matmuls.  Test infrastructure for the library
// (declared in include/attn_fwd_probe.h), not part of the attention path.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "host_util.h"
#include "ptx.cuh"

using namespace attn;

namespace {

constexpr uint64_t kProbeTimeoutNs = 2000000000ull;  // 2 s
constexpr int kTile = 128;

__device__ __forceinline__ uint8_t* align_1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~static_cast<uintptr_t>(1023));
}

// q_rows/k_rows < 128 exercise the zero fill of rows past the end.
__global__ void __launch_bounds__(128, 1)
    probe_mma_ss_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk, int D,
                        float* s_out, uint16_t* q_dump, int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_1024(smem_raw);
  uint8_t* q_s = smem;
  uint8_t* k_s = smem + kTile * D * 2;
  __shared__ uint64_t bar_load, bar_mma;
  __shared__ uint32_t tmem_base;
  __shared__ uint32_t abort_flag;
  const int warp = threadIdx.x / 32;

  if (threadIdx.x == 0) {
    mbar_init(&bar_load, 1);
    mbar_init(&bar_mma, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&tmem_base, 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_base;

  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(&bar_load, 2u * kTile * D * 2);
    for (int c = 0; c < D / 64; ++c) {
      tma_load_3d(q_s + c * kTile * 128, &tq, &bar_load, c * 64, 0, 0);
      tma_load_3d(k_s + c * kTile * 128, &tk, &bar_load, c * 64, 0, 0);
    }
    if (mbar_wait_bounded(&bar_load, 0, &abort_flag, kProbeTimeoutNs)) {
      tc_fence_after();
      const uint32_t idesc = idesc_bf16_f32(128, 128, false);
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk / 4) * (kTile * 128) + (kk % 4) * 32;
        mma_bf16_ss(tbase, sdesc_sw128(smem_u32(q_s) + off, 16, 1024), sdesc_sw128(smem_u32(k_s) + off, 16, 1024),
                    idesc, kk > 0 ? 1u : 0u);
      }
      mma_commit(&bar_mma);
    } else {
      abort_flag = 1;
      atomicExch(status, 1);
    }
  }
  const bool ok = mbar_wait_bounded(&bar_mma, 0, &abort_flag, kProbeTimeoutNs);
  tc_fence_after();
  if (ok) {
    const int row = threadIdx.x;
    for (int c = 0; c < 4; ++c) {
      uint32_t r[32];
      tmem_ld32_wait(tbase + (static_cast<uint32_t>(warp * 32) << 16) + c * 32, r);
      for (int i = 0; i < 32; ++i) s_out[row * kTile + c * 32 + i] = __uint_as_float(r[i]);
    }
  } else if (threadIdx.x == 0) {
    atomicExch(status, 2);
  }
  const uint16_t* qh = reinterpret_cast<const uint16_t*>(q_s);
  for (int i = threadIdx.x; i < kTile * D; i += blockDim.x) q_dump[i] = qh[i];
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tbase, 128);
  }
}

// p: [128][128] bf16 row-major (row = query, column = key); v via map [128][D].
__global__ void __launch_bounds__(128, 1)
    probe_mma_ts_kernel(const __grid_constant__ CUtensorMap tv, const uint32_t* p, int D, uint32_t lbo, uint32_t sbo,
                        float* o_out, int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* v_s = align_1024(smem_raw);
  __shared__ uint64_t bar_load, bar_mma;
  __shared__ uint32_t tmem_base;
  __shared__ uint32_t abort_flag;
  const int warp = threadIdx.x / 32;
  const int row = threadIdx.x;

  if (threadIdx.x == 0) {
    mbar_init(&bar_load, 1);
    mbar_init(&bar_mma, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&tmem_base, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_base;
  const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;

  // P row -> TMEM columns [0, 64): two bf16 per 32-bit column.
  for (int c = 0; c < 2; ++c) {
    uint32_t r[32];
    for (int i = 0; i < 32; ++i) r[i] = p[row * 64 + c * 32 + i];
    tmem_st32(tbase + lane_base + c * 32, r);
  }
  tmem_wait_st();
  tc_fence_before();
  __syncthreads();

  if (threadIdx.x == 0) {
    tc_fence_after();
    mbar_arrive_expect_tx(&bar_load, static_cast<uint32_t>(kTile * D * 2));
    for (int c = 0; c < D / 64; ++c) tma_load_3d(v_s + c * kTile * 128, &tv, &bar_load, c * 64, 0, 0);
    if (mbar_wait_bounded(&bar_load, 0, &abort_flag, kProbeTimeoutNs)) {
      tc_fence_after();
      const uint32_t idesc = idesc_bf16_f32(128, D, true);
      for (int kk = 0; kk < kTile / 16; ++kk)
        mma_bf16_ts(tbase + 128, tbase + kk * 8, sdesc_sw128(smem_u32(v_s) + kk * 16 * 128, lbo, sbo), idesc,
                    kk > 0 ? 1u : 0u);
      mma_commit(&bar_mma);
    } else {
      abort_flag = 1;
      atomicExch(status, 1);
    }
  }
  const bool ok = mbar_wait_bounded(&bar_mma, 0, &abort_flag, kProbeTimeoutNs);
  tc_fence_after();
  if (ok) {
    for (int c = 0; c < D / 32; ++c) {
      uint32_t r[32];
      tmem_ld32_wait(tbase + lane_base + 128 + c * 32, r);
      for (int i = 0; i < 32; ++i) o_out[row * D + c * 32 + i] = __uint_as_float(r[i]);
    }
  } else if (threadIdx.x == 0) {
    atomicExch(status, 2);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tbase, 256);
  }
}

// One warp waits on an mbarrier that nothing ever arrives on, with the same
// bounded wait the attention kernel uses; it must give up after timeout_ns and
// report it (status = 1) instead of hanging.  A second warp raises the abort
// flag instead when abort_after_ns > 0, and the waiter must see it (status = 2).
__global__ void __launch_bounds__(64, 1) probe_wait_timeout_kernel(uint64_t timeout_ns, uint64_t abort_after_ns,
                                                                   int* status, unsigned long long* waited_ns) {
  __shared__ uint64_t bar;
  __shared__ uint32_t abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    const uint64_t t0 = global_timer_ns();
    const bool ok = mbar_wait_bounded(&bar, 0, &abort_flag, timeout_ns);
    const uint64_t t1 = global_timer_ns();
    if (threadIdx.x == 0) {
      *status = ok ? 0 : (abort_flag ? 2 : 1);
      *waited_ns = t1 - t0;
    }
  } else if (abort_after_ns > 0 && threadIdx.x == 32) {
    const uint64_t t0 = global_timer_ns();
    while (global_timer_ns() - t0 < abort_after_ns) {
    }
    *reinterpret_cast<volatile uint32_t*>(&abort_flag) = 1;
  }
  __syncthreads();
}

// Dense bf16 MMA rate: one thread issues n back-to-back tcgen05 MMAs of 128 x N x 16
// (A 128 rows and B N rows, K-major, 128-byte swizzled, zero-filled shared memory),
// accumulating into one TMEM tile, then waits for them; the CTA's clock64 and
// %globaltimer spans give the rate per SM and the clock.  The dynamic shared
// memory keeps one CTA per SM.
__global__ void __launch_bounds__(128, 1) probe_mma_rate_kernel(int n, int N, unsigned long long* cycles,
                                                                unsigned long long* nanos, int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_1024(smem_raw);
  uint8_t* a_s = smem;              // 128 rows x 128 B
  uint8_t* b_s = smem + 128 * 128;  // N rows x 128 B
  __shared__ uint64_t bar_mma;
  __shared__ uint32_t tmem_base;
  __shared__ uint32_t abort_flag;
  const int warp = threadIdx.x / 32;
  for (int i = threadIdx.x; i < (128 + N) * 128 / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    mbar_init(&bar_mma, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&tmem_base, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_base;
  if (threadIdx.x == 0) {
    const uint32_t idesc = idesc_bf16_f32(128, N, false);
    const uint64_t t0 = global_timer_ns();
    const long long c0 = clock64();
    for (int i = 0; i < n; ++i) {
      const uint32_t off = (i % 4) * 32;  // the four K steps of one 128-byte swizzle span
      mma_bf16_ss(tbase, sdesc_sw128(smem_u32(a_s) + off, 16, 1024), sdesc_sw128(smem_u32(b_s) + off, 16, 1024),
                  idesc, i > 0 ? 1u : 0u);
    }
    mma_commit(&bar_mma);
    const bool ok = mbar_wait_bounded(&bar_mma, 0, &abort_flag, kProbeTimeoutNs);
    const long long c1 = clock64();
    const uint64_t t1 = global_timer_ns();
    cycles[blockIdx.x] = static_cast<unsigned long long>(c1 - c0);
    nanos[blockIdx.x] = t1 - t0;
    if (!ok) atomicExch(status, 2);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tbase, 256);
  }
}

// ex2.approx rate: every thread runs 8 independent chains x <- 2^x - 1.5 (the
// subtraction, on the FMA pipe, keeps x bounded), `iters` steps each.
__global__ void __launch_bounds__(512, 1) probe_ex2_rate_kernel(int iters, unsigned long long* cycles,
                                                                float* sink) {
  float x[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) x[c] = 0.01f * (threadIdx.x % 7) + 0.1f * c;
  __syncthreads();
  const long long c0 = clock64();
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int c = 0; c < 8; ++c) x[c] = ex2_approx(x[c]) - 1.5f;
  }
  __syncthreads();
  const long long c1 = clock64();
  float acc = 0.0f;
#pragma unroll
  for (int c = 0; c < 8; ++c) acc += x[c];
  sink[blockIdx.x * blockDim.x + threadIdx.x] = acc;
  if (threadIdx.x == 0) cycles[blockIdx.x] = static_cast<unsigned long long>(c1 - c0);
}

int launch_status(cudaError_t e) { return e == cudaSuccess ? 0 : 100 + static_cast<int>(e); }

}  // namespace

extern "C" {

int attn_probe_mma_ss(const void* q, int q_rows, const void* k, int k_rows, int D, float* s_out, void* q_dump,
                      int* status, cudaStream_t stream) {
  if (!q || !k || !s_out || !q_dump || !status) return 2;
  if ((D != 64 && D != 128) || q_rows < 1 || q_rows > kTile || k_rows < 1 || k_rows > kTile) return 1;
  CUtensorMap tq, tk;
  if (!attn_host::encode_bf16_rows(&tq, q, D, q_rows, 1, kTile)) return 3;
  if (!attn_host::encode_bf16_rows(&tk, k, D, k_rows, 1, kTile)) return 3;
  const int smem = 2 * kTile * D * 2 + 1024;
  cudaError_t e = cudaFuncSetAttribute(probe_mma_ss_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return launch_status(e);
  probe_mma_ss_kernel<<<1, 128, smem, stream>>>(tq, tk, D, s_out, static_cast<uint16_t*>(q_dump), status);
  return launch_status(cudaGetLastError());
}

int attn_probe_mma_ts(const void* p, const void* v, int D, int lbo, int sbo, float* o_out, int* status,
                      cudaStream_t stream) {
  if (!p || !v || !o_out || !status) return 2;
  if (D != 64 && D != 128) return 1;
  if (lbo < 0 || sbo < 0 || lbo > 65535 || sbo > 65535 || (lbo % 16) || (sbo % 16)) return 1;
  CUtensorMap tv;
  if (!attn_host::encode_bf16_rows(&tv, v, D, kTile, 1, kTile)) return 3;
  const int smem = kTile * D * 2 + 1024;
  cudaError_t e = cudaFuncSetAttribute(probe_mma_ts_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return launch_status(e);
  probe_mma_ts_kernel<<<1, 128, smem, stream>>>(tv, static_cast<const uint32_t*>(p), D, static_cast<uint32_t>(lbo),
                                                static_cast<uint32_t>(sbo), o_out, status);
  return launch_status(cudaGetLastError());
}

int attn_probe_wait_timeout(unsigned long long timeout_ns, unsigned long long abort_after_ns, int* status,
                            unsigned long long* waited_ns, cudaStream_t stream) {
  if (!status || !waited_ns) return 2;
  if (timeout_ns == 0 || timeout_ns > 2000000000ull || abort_after_ns > 2000000000ull) return 1;
  probe_wait_timeout_kernel<<<1, 64, 0, stream>>>(timeout_ns, abort_after_ns, status, waited_ns);
  return launch_status(cudaGetLastError());
}

int attn_probe_mma_rate(int n_mma, int N, int grid, unsigned long long* cycles, unsigned long long* nanos,
                        int* status, cudaStream_t stream) {
  if (!cycles || !nanos || !status) return 2;
  if (n_mma < 1 || n_mma > (1 << 20) || (N != 64 && N != 128 && N != 256) || grid < 1 || grid > 1024) return 1;
  const int smem = 200 * 1024;  // one CTA per SM (the operands need 48 KB at most)
  cudaError_t e = cudaFuncSetAttribute(probe_mma_rate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return launch_status(e);
  probe_mma_rate_kernel<<<grid, 128, smem, stream>>>(n_mma, N, cycles, nanos, status);
  return launch_status(cudaGetLastError());
}

int attn_probe_ex2_rate(int iters, int grid, unsigned long long* cycles, float* sink, cudaStream_t stream) {
  if (!cycles || !sink) return 2;
  if (iters < 1 || iters > (1 << 20) || grid < 1 || grid > 1024) return 1;
  probe_ex2_rate_kernel<<<grid, 512, 0, stream>>>(iters, cycles, sink);
  return launch_status(cudaGetLastError());
}

}  // extern "C"
