/*
 * pa_probe.h -- measurement and test aids, not part of the attention path;
 * the pages have no counterpart for them. They live in their own library,
 * libpa_probe.so, next to libpa.so.
 *
 * pa_gather_probe streams whole K and V blocks of a paged pool into shared
 * memory with the same machinery the decode kernel uses (persistent CTAs, a
 * ring of `stages` bulk-copy stages completed on mbarriers, one 1-D copy per
 * block and pool) and computes nothing. The time it takes bounds what the
 * decode kernel can reach on the same block list: the gap between the two is
 * spent on the SMs, not on HBM.
 *
 *  pool      the pool (pa.h); only its pointers, sizes and dtype are used
 *  blocks    device int32 [n], physical block ids (each in [0, num_blocks))
 *  stages    1..8 stages of one K block + one V block each; the stages must
 *            fit in 227 KB of shared memory
 *  ctas      persistent CTAs (0: one per SM); CTA c streams blocks
 *            [c*n/ctas, (c+1)*n/ctas)
 *  d_status  device int, nullable: PA_STATUS_BAD_BLOCK for an id outside
 *            the pool (skipped), PA_STATUS_TIMEOUT if a copy never completed
 *
 * Asynchronous on `stream`; returns a pa_status.
 */
#ifndef PA_PROBE_H
#define PA_PROBE_H

#include <stdint.h>

#include "pa.h"

#ifdef __cplusplus
extern "C" {
#endif

PA_API int pa_gather_probe(const pa_kv_pool* pool, const int32_t* blocks, int n, int stages,
                           int ctas, int* d_status, void* stream);

/*
 * pa_wait_probe runs, in one CTA, the bounded wait and give-up path that every
 * libpa kernel takes when an asynchronous copy does not complete, without
 * leaving anything in flight: a warp holds 32 TMEM columns, thread 0 arms an
 * mbarrier for a 1,024-byte bulk copy, and every thread waits on it for at
 * most limit_ns of global time.
 *
 *  src       device, 16-byte aligned, >= 1,024 bytes: the copy's source
 *  starve    0: the copy is issued, the wait completes, the copied bytes are
 *            checked (PA_STATUS_BAD_BLOCK on a mismatch);
 *            1: the barrier is armed but the copy never started, so the wait
 *            runs out: the kernel ORs PA_STATUS_TIMEOUT into *d_status,
 *            releases its TMEM and returns
 *  limit_ns  1 .. 2e9 (the kernels' own limit); PA_EINVAL otherwise
 *  d_status  device int, nullable
 *
 * Asynchronous on `stream`; returns a pa_status.
 */
PA_API int pa_wait_probe(const void* src, int starve, unsigned long long limit_ns, int* d_status,
                         void* stream);

#ifdef __cplusplus
}
#endif
#endif /* PA_PROBE_H */
