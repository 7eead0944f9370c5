/*
 * cpa_test.h -- test hooks of the checked build of the library
 * (libcpa_checked.so, compiled with CPA_BOUNDS_CHECK and CPA_TEST_HOOKS).
 *
 * The pages have no counterpart: these exist so that the failure paths of
 * the kernels can be exercised without faulting a GPU.  In the checked build
 * every in-kernel pipeline wait gives up after 20 ms (200 ms in the library)
 * and every index the kernels compute for a global access is range-checked
 * (an index outside its buffer sets CPA_EBIT_BOUNDS and the access is
 * skipped).  The regular library (libcpa.so) does not export this symbol.
 */
#ifndef CPA_TEST_H_
#define CPA_TEST_H_

#include "cpa.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * From the next attention call on, the K/V producer of the two-tile kernel
 * issues no copy for the `tile`-th key tile of each CTA (counted from 0 over
 * the CTA's whole walk); -1 (the default) withholds nothing.  The consumer's
 * bounded wait for that tile then runs out: the CTA stops its roles, lets
 * every copy and product in flight finish, frees its tensor memory and sets
 * CPA_EBIT_TIMEOUT in the call's error word.  The outputs of such a call are
 * undefined.  Host-side setting, read when a call is launched; not thread
 * safe.
 */
void cpa_test_drop_tile(int tile);

#ifdef __cplusplus
}
#endif

#endif /* CPA_TEST_H_ */
