/*
 * exq_testing.h -- test hook of libexq for failure detection. It has no
 * counterpart in the ExLlamaV2 pages: it exists so that a test can watch a
 * bounded device-side wait give up without faulting, trapping or hanging
 * the GPU.
 */
#ifndef EXQ_TESTING_H
#define EXQ_TESTING_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* exq_testing_starve -- while wait_rounds > 0, every exq_gemv, exq_gemv_multi
 * and exq_gemm launch runs with its producer issuing no copies at all, and
 * every mbarrier wait of those kernels gives up after wait_rounds polling
 * rounds instead of the built-in bound. The consumers then wait for data that
 * never comes; their bounded waits run out, the kernel records
 * EXQ_ERR_TIMEOUT in the device error word (read it with
 * exq_get_last_device_error), frees what it holds (tensor memory) and
 * returns. No copy is in flight at any time, so nothing is left to drain.
 * Outputs of a starved call are unspecified; a starved exq_gemv may leave its
 * workspace counters non-zero (zero them before the next call).
 * wait_rounds = 0 turns the hook off (the default). Host-side, process-wide,
 * thread-safe; it affects launches made after it returns. */
void exq_testing_starve(int32_t wait_rounds);

#ifdef __cplusplus
}
#endif

#endif /* EXQ_TESTING_H */
