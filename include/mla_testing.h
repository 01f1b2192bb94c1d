/*
 * mla_testing.h - test hooks of the MLA library (not part of the decode path).
 *
 * They let the test-suite exercise the library's failure handling on a GPU
 * without faulting, trapping or hanging it.
 */
#ifndef MLA_TESTING_H_
#define MLA_TESTING_H_

#include "mla.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * mla_test_bounded_wait - enqueue one tiny kernel whose thread waits on an
 * on-chip barrier that nothing ever completes, using the same bounded-wait
 * routine as the decode kernels but with a limit of `limit_ms` milliseconds
 * (1..10000).  The wait gives up, the kernel records MLA_DEV_WAIT_TIMEOUT in
 * the device status word and returns normally; the CUDA context stays usable.
 * Read the result with mla_get_device_status().
 */
mla_status_t mla_test_bounded_wait(int limit_ms, mla_stream_t stream);

/*
 * mla_test_launch_count - number of kernels the library has enqueued in this
 * process so far, on any device and stream (every successful launch of every
 * entry point counts one; host-side argument errors launch and count nothing).
 * Host only, thread-safe.  Lets a benchmark count the kernels of a timed region
 * (read it before and after) rather than assume them.
 */
uint64_t mla_test_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* MLA_TESTING_H_ */
