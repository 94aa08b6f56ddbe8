/*
 * osr_test.h -- test support of the GB300 row-wise reduce-then-rescale
 * library.  These entry points exist so that tests can reach internals the
 * computation itself never exposes; no computation path calls them, and
 * the operations they serve have no counterpart on the pages the library
 * follows.
 */
#ifndef OSR_TEST_H
#define OSR_TEST_H

#include <stdint.h>

#include "osr.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Test flags applied to every later launch of the calling process, until
 * set again (0 = none).  Bit 0 (OSR_TEST_NO_ARRIVE): the staged softmax
 * tier's copy barrier receives no arrival, so its bounded wait runs out
 * (about 1 s) and the kernel reports the fault through osr_device_fault
 * instead of computing.  Returns the previous flags.
 */
#define OSR_TEST_NO_ARRIVE 1
int osr_test_set_flags(int flags);

/*
 * Force the dispatcher's choice for every later call of the calling process
 * (compute entry points and osr_plan_describe alike) until cleared with
 * NULL or "".  The spec names a tier and its shape, e.g. "rows:g=512",
 * "cluster:g=256,cs=2", "staged:cs=3,r=8", "split:s=7,b=3", "lse:cs=4,st=0",
 * "lse:g=32", "topk:cs=8"; a shape the tier cannot take makes the calls
 * return OSR_ERR_UNSUPPORTED.  The spec is copied (at most 63 characters,
 * else OSR_ERR_INVALID).  Tests use it to run every tier on chosen shapes;
 * with none set the planners read nothing but an atomic flag.
 */
osr_status osr_test_force_kernel(const char *spec);

/*
 * The kernels' e^(x - m), evaluated on the device beside CUDA's expf, so a
 * test can hold it to its error bound.  For i < n:
 *   approx[i] = the library's e^(x[i] - m[i]): (x - m) * log2(e) rounded
 *               to binary32, then the ex2.approx.ftz special-function
 *               instruction (results below 2^-126 flush to 0);
 *   ref[i]    = expf(x[i] - m[i]) (CUDA's binary32 exponential).
 * x, m, approx, ref: device pointers to n floats (caller-owned).
 * Asynchronous on `stream`; OSR_ERR_INVALID for n < 0 or a NULL pointer,
 * OSR_ERR_CUDA if the launch fails.
 */
osr_status osr_test_exp_shifted(const float *x, const float *m, float *approx, float *ref,
                                int64_t n, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* OSR_TEST_H */
