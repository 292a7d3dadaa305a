/*
 * attn_fwd_probe.h -- primitive checks of the building blocks of the attention
 * kernel, exported by libattn_probe.so.  Test infrastructure: each entry point
 * runs one CTA on one 128-row tile so a CPU matmul can check the hand-encoded
 * TMA tensor maps, shared-memory descriptors, instruction descriptors and
 * tensor-memory access patterns the attention kernel relies on.  They have no
 * counterpart on the pages; they exist because the compiled code itself may
 * not be inspected.
 *
 * Every pointer is device memory; calls are asynchronous on `stream`.
 * Return: 0 when launched; 1 bad size; 2 NULL pointer; 3 tensor map rejected;
 * 100 + cudaError_t when a CUDA call failed.  `status` (one int, zeroed by the
 * caller) receives 1 or 2 if a wait inside the kernel ran out of time.
 */
#ifndef ATTN_FWD_PROBE_H
#define ATTN_FWD_PROBE_H

#include <cuda_runtime.h>

#ifdef __cplusplus
extern "C" {
#endif

/*
 * S = Q K^T for one tile.  q: [q_rows][D] bf16, k: [k_rows][D] bf16 with
 * 1 <= q_rows, k_rows <= 128 (rows past the end read as zero through TMA).
 * s_out: [128][128] fp32 row-major.  q_dump: [128 * D] bf16 receives the raw
 * (swizzled) shared-memory image of the Q tile as TMA wrote it.
 */
int attn_probe_mma_ss(const void* q, int q_rows, const void* k, int k_rows, int D, float* s_out, void* q_dump,
                      int* status, cudaStream_t stream);

/*
 * O = P V for one tile with P taken from tensor memory.  p: [128][128] bf16
 * (row = query, column = key), written into tensor memory with tcgen05.st;
 * v: [128][D] bf16 loaded by TMA (MN-major operand).  lbo/sbo: the leading-
 * and stride-dimension byte offsets put into V's shared-memory descriptor.
 * o_out: [128][D] fp32 row-major.
 */
int attn_probe_mma_ts(const void* p, const void* v, int D, int lbo, int sbo, float* o_out, int* status,
                      cudaStream_t stream);

/*
 * Failure handling of the bounded waits, without faulting or hanging the GPU:
 * one warp waits on an mbarrier that nothing arrives on, using the wait the
 * attention kernel uses.  It must give up after timeout_ns (1 ns .. 2 s) and
 * write *status = 1, or, when abort_after_ns > 0, see the abort flag another
 * warp raises after that time and write *status = 2.  *waited_ns receives how
 * long the wait lasted (device %globaltimer).  status, waited_ns: device memory.
 */
int attn_probe_wait_timeout(unsigned long long timeout_ns, unsigned long long abort_after_ns, int* status,
                            unsigned long long* waited_ns, cudaStream_t stream);

/*
 * Dense bf16 tensor-core rate: `grid` CTAs (one per SM) each issue n_mma
 * back-to-back tcgen05 MMAs of 128 x N x 16 (N = 64, 128 or 256) from one
 * thread into one TMEM accumulator and wait for them.  cycles[c] / nanos[c]
 * (device memory, `grid` entries each) receive CTA c's clock64 and %globaltimer
 * spans: 2 * 128 * N * 16 * n_mma / cycles is the dense bf16 FLOP per clock of an
 * SM, cycles / nanos its clock in GHz.  *status = 2 if the wait ran out.
 */
int attn_probe_mma_rate(int n_mma, int N, int grid, unsigned long long* cycles, unsigned long long* nanos,
                        int* status, cudaStream_t stream);

/*
 * ex2.approx rate: `grid` CTAs of 512 threads, each thread running 8
 * independent exponential chains for `iters` steps.  cycles[c] receives CTA
 * c's clock64 span, so 512 * 8 * iters / cycles is the exponentials per clock of
 * an SM (with one CTA per SM).  sink: grid * 512 floats (keeps the chains).
 */
int attn_probe_ex2_rate(int iters, int grid, unsigned long long* cycles, float* sink, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_FWD_PROBE_H */
