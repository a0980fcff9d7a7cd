/*
 * test_hooks.h -- the one extra symbol of libloom_test.so, a build of libloom
 * for the fault tests (the same kernels; the host layer compiled with
 * LOOM_TEST_HOOKS).  The shipping libloom.so does not export it.
 */
#ifndef LOOM_TEST_HOOKS_H
#define LOOM_TEST_HOOKS_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* While `on` is non-zero, every staged kernel launched by this process issues
 * no copies, so each of its waits runs out after the tuning's wait limit
 * (loom_tuning.wait_ns): the results become NaN, the error word gets
 * LOOM_DEVERR_TIMEOUT, and the device stays usable.  Process-wide. */
void loom_test_inject_stall(int32_t on);

#ifdef __cplusplus
}
#endif

#endif /* LOOM_TEST_HOOKS_H */
