/*
 * attn_fwd_trace.h -- timeline of the forward kernel, in the library built with
 * -DATTN_TRACE (libattn_fwd_trace.so; the default libattn_fwd.so has none of it).
 *
 * The traced library exports everything attn_fwd.h declares, computing the same
 * results bit for bit, and records in device memory, for each CTA c < 160 and
 * each role, up to 2048 events of its launches as (t, code, arg): t the
 * %globaltimer value in ns when lane 0 of the role's warp reached the point.
 * Roles: 0 TMA producer, 1 tcgen05 issuer, 2 softmax of Q tile 0 (warp 0),
 * 3 softmax of Q tile 1 (warp 4), 4 O store warp.  Events:
 *     0  CTA start (producer)                 1  item published (arg: item, -1 = none left)
 *     2  K tile load issued (arg: key tile)   3  V tile load issued (arg: key tile)
 *    12  item's first S products issued (arg: item)
 *    11  P.V issued (arg: Q tile)            13  every MMA of the CTA completed
 *    22  the thread's share of V_j converted to fp16 (arg: j, the item's tile number)
 *    20  S_t(j) ready to read (arg: j)       21  P_t(j) handed to the MMA (arg: j)
 *    23  O_t read out of tensor memory (arg: item)
 *    24  O_t staged for its TMA store (arg: item)
 *    30  O stores of Q tile t issued (arg: t)   31  every store landed (store warp's end)
 * The recording adds a global store and a timer read per event to each role,
 * so timings come out longer than in the default build (the softmax's own
 * events, two per key tile, lengthen the train workload's launch by about a
 * seventh); events finer than these were tried and distorted the timeline.
 */
#ifndef ATTN_FWD_TRACE_H
#define ATTN_FWD_TRACE_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Synchronise the device, copy the recorded events of the launches since the
 * previous read into `dst` (host memory) and clear the event counts.  Layout of
 * `dst`: uint32 count[ctas][roles] (events a role reached; more than `events`
 * means the later ones were not kept), then records[ctas][roles][events] of
 * { uint64 t; uint32 code; uint32 arg; }.  `ctas`, `roles`, `events` (each may be
 * NULL) receive the array sizes.  Returns ATTN_OK, ATTN_ERR_NULL_PTR,
 * ATTN_ERR_INVALID_ARG when `dst_bytes` is too small for both arrays, or
 * ATTN_ERR_CUDA.
 */
int attn_fwd_trace_read(void* dst, size_t dst_bytes, int* ctas, int* roles, int* events);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_FWD_TRACE_H */
