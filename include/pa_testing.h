/*
 * pa_testing.h -- test hooks of libpa.  Not part of the paged-attention
 * boundary (include/pa.h) and not meant for production callers; the pages
 * have no counterpart.
 *
 * Every pipeline wait inside the bf16 and FP8 decode kernels (a consumer
 * waiting for a copy to land, a producer waiting for a stage to be freed)
 * is bounded: after a number of polls it gives up, sets
 * PA_DEVERR_TIMEOUT in the device error word, lets the CTA's own copies in
 * flight land (those waits keep their own bound), and returns.  A correct
 * pipeline never comes near the bound, so tests need a way to make a wait
 * run out on purpose without faulting or hanging the GPU.
 */
#ifndef PA_TESTING_H_
#define PA_TESTING_H_

#include <stdint.h>

#include "pa.h"

#ifdef __cplusplus
extern "C" {
#endif

/* pa_testing_set_wait_limit -- process-wide; applies to decode calls
 * (pa_decode, pa_decode_append, pa_decode_append_fp8, pa_decode_cascade's
 * suffix pass, pa_decode_noalloc) launched after it returns.
 *   polls  polls before a wait of the math warp (the only warp of an FP8
 *          CTA) gives up; 0 restores the default (2^22) and clears
 *          `stall`.  The copy warp of a bf16 CTA always uses the default,
 *          so after a stalled math warp it gives up later.
 *   stall  1: the math warp of every decode CTA first waits on a barrier
 *          that nothing arrives at, with the limit above, so that wait runs
 *          out deterministically: the CTA sets PA_DEVERR_TIMEOUT, drains its
 *          copies and exits without writing its part of the output.
 *          0: normal operation with the given limit.
 * Returns PA_ERR_INVALID_ARG for a stall value other than 0 or 1.  The
 * NVFP4 decode kernels have no mbarrier waits and ignore both settings. */
pa_status pa_testing_set_wait_limit(uint32_t polls, int32_t stall);

#ifdef __cplusplus
}
#endif

#endif  /* PA_TESTING_H_ */
