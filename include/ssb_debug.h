/* Test hooks of libssb: entry points that the library's own tests call to reach code paths
 * that ordinary inputs do not exercise.  They are exported with the C ABI of ssb.h, take
 * the same plain pointers, sizes and status codes, and never trap the GPU.  They are not
 * meant for production use.
 */
#ifndef SSB_DEBUG_H
#define SSB_DEBUG_H

#include <stddef.h>

#include "ssb.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Bounded-wait failure path.  In the next library call on c that evaluates the objective
 * (ssb_loss_batch, ssb_reconstruct, ssb_reconstruct_upsampled, ssb_profile_objective),
 * evaluation number `evaluation` (0 = the first trial of the call) makes its row tasks
 * wait for a completion count that nothing ever reaches, with a poll limit of `polls`
 * (0 is taken as 1).  The wait then gives up, raises the kernel's error word, every other
 * wait stops, the kernel returns, and the call reports SSB_ERR_TIMEOUT; the losses of that
 * trial and of every later trial of the call are NaN (and so may be the loss of the trial
 * before it, whose launch overlaps it on the GPU).  The hook is consumed by that call.
 * This is the timeout behaviour of the boundary (status codes only, no trap); the pages
 * define no counterpart.  NULL c or evaluation < 0 -> SSB_ERR_ARG. */
ssb_status ssb_debug_stall_next(ssb_ctx *c, int evaluation, unsigned polls);

/* Fill every per-evaluation scratch buffer of c (the column-to-row ring and its Nyquist
 * terms, the accumulators, the per-trial tables, the scheduler words and the loss slots)
 * with 0xFF bytes (NaN as float) on cuda_stream, then synchronise it.  A following call
 * must give the same results bit for bit as without the poison: every value the objective
 * reads was written by that evaluation.  This is the pages' phase-only against
 * phase-plus-loss bit-identity check that exposed unwritten rows ("SSB performance notes",
 * MPS wider exact-simplex checkpoint), made stronger.  NULL c -> SSB_ERR_ARG. */
ssb_status ssb_debug_poison_scratch(ssb_ctx *c, void *cuda_stream);

/* out[i] = the objective's float32 phase function atan2(y[i], x[i]) in (-pi, pi], for n
 * elements of device arrays (float32), on cuda_stream, which it synchronises.  The phase
 * phi_k(r) = atan2(Im c_k, Re c_k) is step 6 of the objective (the per-BF phase of the
 * corrected image before the moments).  n = 0 is a no-op; NULL pointers with n > 0 ->
 * SSB_ERR_ARG. */
ssb_status ssb_debug_atan2(const float *y_device, const float *x_device, size_t n,
                           float *out_device, void *cuda_stream);

#ifdef __cplusplus
}
#endif
#endif /* SSB_DEBUG_H */
