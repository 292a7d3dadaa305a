/*
 * attn_bwd_trace.h -- timeline of the backward kernels, in the library built with
 * -DATTN_TRACE (libattn_bwd_trace.so; the default libattn_bwd.so has none of it).
 *
 * The traced library exports everything attn_bwd.h declares, computing the same
 * gradients bit for bit, and records in device memory, for each of the two main
 * kernels (0: dK/dV, 1: dQ), each CTA c < 160 and each role, up to 2048 events of
 * its launches as (t, code, arg): t the %globaltimer value in ns when lane 0 of
 * the role's first warp reached the point.  Roles: 0 TMA producer, 1 tcgen05
 * issuer, 2 compute warpgroup 0 (warp 0), 3 compute warpgroup 1 (warp 4).
 * Events:
 *      0  CTA start (producer)
 *      1  the item's fixed tiles requested (arg: item): K and V (dK/dV), Q and dO (dQ)
 *     10  the item's first S-type products issued (arg: item)
 *     11  the first of a step's two accumulating products issued: dV and dK of half 0
 *         (dK/dV; arg: the step's index within its item), dQ += dS K of keys 0-63 (dQ;
 *         arg: bit 0 set unless it is the item's first step, bit 1 set on its last)
 *     13  every MMA of the CTA completed (issuer's end)
 *     20  the step's S-type products ready to read (arg: step within the item)
 *     21  the warpgroup's P and dS handed to the MMA (arg: step within the item)
 *     23  the item's accumulators complete: its epilogue starts (arg: item)
 *     24  the epilogue has read the accumulators and stored the rows (arg: item)
 * The recording adds a global store and a timer read per event to each role, so
 * timings come out somewhat longer than in the default build.
 */
#ifndef ATTN_BWD_TRACE_H
#define ATTN_BWD_TRACE_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Synchronise the device, copy the recorded events of the launches since the
 * previous read into `dst` (host memory) and clear the event counts.  Layout of
 * `dst`: uint32 count[kernels][ctas][roles] (events a role reached; more than
 * `events` means the later ones were not kept), then
 * records[kernels][ctas][roles][events] of { uint64 t; uint32 code; uint32 arg; }.
 * `kernels`, `ctas`, `roles`, `events` (each may be NULL) receive the array sizes.
 * Returns ATTN_OK, ATTN_ERR_NULL_PTR, ATTN_ERR_INVALID_ARG when `dst_bytes` is
 * too small for both arrays, or ATTN_ERR_CUDA.
 */
int attn_bwd_trace_read(void* dst, size_t dst_bytes, int* kernels, int* ctas, int* roles, int* events);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_BWD_TRACE_H */
