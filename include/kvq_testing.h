/*
 * kvq_testing.h -- test hooks of the kvq library.  Not part of the method:
 * the pages have no counterpart; these exist so that the failure paths of the
 * decode kernel can be exercised without faulting or hanging a GPU.
 *
 * Every wait of the decode kernel on a shared-memory copy is bounded: when it
 * runs out, the warp sets KVQ_FLAG_TIMEOUT in the cache's status word, lets
 * its copies still in flight land (each wait again bounded) and returns, so
 * the context stays usable and kvq_get_device_status() reports
 * KVQ_ERR_TIMEOUT.  The hook below makes one such wait run out on purpose.
 */
#ifndef KVQ_TESTING_H
#define KVQ_TESTING_H

#include <stdint.h>

#include "kvq.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * kvq_testing_set_decode_fault -- settings of every later multi-head decode
 * launch of this process (kvq_decode_attention, _noalloc, _gqa with one query
 * head per cache head, and such steps captured into a graph after the call),
 * on every device, until changed again; while they differ from the defaults
 * those launches run an instantiation of the kernel that reads them:
 *   wait_limit_us  limit of each bounded wait in microseconds; 0 restores the
 *                  default of 0.5 s
 *   skip_chunk     >= 0: the first warp of the grid arms the barrier of its
 *                  chunk number skip_chunk (0 = the first stage it fills) but
 *                  issues none of that chunk's copies, so its wait for the
 *                  chunk runs out with nothing in flight; -1 (the default)
 *                  turns this off.  A chunk number the warp never reaches
 *                  changes nothing.
 * After a launch that timed out, the split counters of its workspace are left
 * non-zero: zero-fill the workspace before reusing it (later calls on it
 * otherwise report KVQ_FLAG_BAD_WORKSPACE).  Errors: KVQ_ERR_INVALID_ARG for
 * skip_chunk < -1.
 */
kvq_status kvq_testing_set_decode_fault(uint32_t wait_limit_us, int32_t skip_chunk);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_TESTING_H */
