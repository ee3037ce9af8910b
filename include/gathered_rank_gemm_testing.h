/*
 * gathered_rank_gemm — test hooks.  Not part of the operation's contract:
 * these calls exist so that the error paths of the kernels can be exercised
 * on a working GPU without faulting it or hanging it.
 */
#ifndef GATHERED_RANK_GEMM_TESTING_H
#define GATHERED_RANK_GEMM_TESTING_H

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Makes the kernels' bounded waits run out, on purpose and quickly.  While
 * `on` is non-zero, every shrink, expand and fused kernel enqueued afterwards
 * (by any entry point) arms the first barrier it waits on with one arrival
 * more than any thread makes, issues no copy into shared memory, and gives a
 * wait up after 1 ms instead of 200 ms.  Each CTA with work then gives up its
 * first wait, every later wait at once, writes no output, waits for nothing
 * in flight (it issued nothing) and ORs LORA_STATUS_TIMEOUT into the status
 * word: the call leaves u and y as they were.  The grouping kernel has no
 * such wait and runs as usual.  The switch is process-wide and read when a
 * launch is enqueued (a CUDA graph keeps the value it was captured with).
 * Returns the previous setting.  Thread-safe; makes no GPU call.
 *
 * The same code paths serve a real timeout: a CTA whose wait runs out stops
 * issuing copies and storing outputs, waits (bounded) for the copies it had
 * issued, and reports LORA_STATUS_TIMEOUT; the outputs of such a call are
 * unspecified.
 */
int lora_testing_inject_timeout(int on);

#ifdef __cplusplus
}
#endif

#endif /* GATHERED_RANK_GEMM_TESTING_H */
