/*
 * eagle3_testing.h - test hooks of libeagle3 (not part of the draft-and-verify step).
 *
 * Every wait inside the library's kernels is bounded: when it runs out the kernel sets
 * EAGLE3_DEV_TIMEOUT in the caller's dev_status word, drains the copies it has in flight, frees
 * its tensor memory and returns, so the CUDA context stays usable (see eagle3.h).  In correct code
 * no wait runs out, so that path only runs when a wait is made to run out on purpose: this hook
 * does that without faulting or hanging anything.
 */
#ifndef EAGLE3_TESTING_H
#define EAGLE3_TESTING_H

#include "eagle3.h"

#ifdef __cplusplus
extern "C" {
#endif

/* eagle3_test_verify_attn_timeout - eagle3_verify_attn (same arguments and workspace) with two
 * changes: the prefix K tile `stall_tile` (counted from the first tile of each CTA's split, so 0 is
 * the first) is never loaded, and every bounded wait gives up after `wait_limit_cycles` SM clocks
 * instead of about two seconds.  Each CTA with more than stall_tile prefix tiles therefore waits
 * for a tile that never arrives, gives up, sets EAGLE3_DEV_TIMEOUT and exits cleanly; its output
 * rows are void.  No counterpart on the pages: it exists to test the failure path.
 * Returns EAGLE3_ERR_INVALID_ARGUMENT for stall_tile < 0 or wait_limit_cycles outside
 * [1000, 4e9], otherwise what eagle3_verify_attn returns. */
eagle3_status_t eagle3_test_verify_attn_timeout(const eagle3_verify_attn_args_t *args, void *workspace,
                                                size_t workspace_bytes, int32_t stall_tile,
                                                int64_t wait_limit_cycles, eagle3_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* EAGLE3_TESTING_H */
