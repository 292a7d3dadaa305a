/*
 * attn_bwd.h -- C ABI of the backward of the exact attention forward pass for
 * GB300 (sm_103a): the gradients of O = softmax(scale * Q K^T + mask) V (see
 * attn_fwd.h for the forward, its masks, layouts and grouped heads) with respect
 * to Q, K and V, for an upstream gradient dO and the forward's saved O and LSE.
 *
 * Operation.  With P_ij = exp(scale q_i.k_j - LSE_i) over the keys row i sees:
 *     dV_j  = sum_i P_ij dO_i                     (sum over every query head of the kv head)
 *     dP_ij = dO_i . v_j,   D_i = dO_i . O_i,   dS_ij = P_ij (dP_ij - D_i)
 *     dQ_i  = scale sum_j dS_ij k_j
 *     dK_j  = scale sum_i dS_ij q_i               (sum over every query head of the kv head)
 * This is the gradient of the softmax attention with a closed-form log-sum-exp
 * normaliser of page "AdaSplash-2: Faster Differentiable Sparse Attention"
 * (technical summary section 1), whose summary notes the backward pass visits
 * only the blocks it needs: under a causal mask no tile wholly above the
 * diagonal is loaded.  No gradient flows in through the LSE.
 *
 * Layout (contiguous, row-major, device memory, 16-byte aligned):
 *     q, o, dout, dq [B][Hq][Sq][D] bf16    k, v, dk, dv [B][Hkv][Sk][D] bf16
 *     lse [B][Hq][Sq] fp32 (the forward's)  workspace: attn_bwd_workspace_size bytes
 * D is 64 or 128; Hq a multiple of Hkv; scale finite and positive (the
 * forward's); causal as in attn_fwd (0, 1 bottom-right, 2 top-left).  Rows without keys get dq = 0; keys no row sees get dk = dv = 0.
 *
 * Precision.  bf16 inputs; S, dP and the three gradients accumulate in fp32 on
 * the tensor cores; P and dS are rounded to bf16 before the products that use
 * them; D_i is formed in fp32 from the bf16 O and dO; the gradients are rounded
 * to bf16 once, at the end.
 *
 * Ownership and execution.  The caller owns every buffer; dq, dk, dv and the
 * workspace must not overlap each other or any input.  Three kernels are
 * enqueued on `stream`; nothing is allocated and nothing is synchronised.
 * Status codes are attn_fwd.h's ATTN_* codes.
 */
#ifndef ATTN_BWD_H
#define ATTN_BWD_H

#include <cuda_runtime.h>
#include <stddef.h>

#include "attn_fwd.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Enqueue the backward pass.  Argument checks run on the host before any device
   work.  B == 0 returns ATTN_OK without work; Sq == 0 or Sk == 0 only zero the
   gradients that exist. */
int attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
             void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Sq, int Sk, int D, int causal, float scale,
             void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Workspace bytes attn_bwd needs: two fp32 values per query row, rows padded to a
   multiple of 128 per (batch, head); 0 for invalid sizes.  Host only. */
size_t attn_bwd_workspace_size(int B, int Hq, int Sq);

/* Text for a status code (ATTN_ERR_CUDA names this library's last CUDA error on the
   calling thread). */
const char* attn_bwd_strerror(int status);

/* Synchronise `stream`, then read and clear the backward kernels' device status
   word (set when one of their bounded waits ran out): ATTN_OK,
   ATTN_ERR_DEVICE_TIMEOUT or ATTN_ERR_CUDA.  `site` (may be NULL) receives it. */
int attn_bwd_debug_status(cudaStream_t stream, int* site);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_BWD_H */
