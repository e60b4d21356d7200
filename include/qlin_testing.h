/*
 * qlin_testing.h -- entry points of libqlin that exist only so that the
 * library's own tests can reach failure paths without faulting or hanging a
 * GPU.  They have no counterpart on the pages the method comes from, and no
 * product code calls them.
 */
#ifndef QLIN_TESTING_H_
#define QLIN_TESTING_H_

#include "qlin.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * qlin_qmv_chain with one dependency that can never be met: the links that
 * read link `stalled_link` wait for one more completed row block than that
 * link has, so their bounded wait runs out after `wait_limit_us`
 * microseconds (1 .. 2,000,000).  The kernel then records bit 2 of the chain
 * kernel's status (qlin_device_status reports 1 << 18), carries on with
 * whatever the input holds (those outputs are garbage), lets every bulk copy
 * it issued land, and exits; the context stays usable.  Arguments otherwise
 * as qlin_qmv_chain.  Errors: QLIN_ERR_INVALID_ARG when stalled_link is out of
 * range or no later link reads it, or wait_limit_us is out of range; else as
 * qlin_qmv_chain.
 */
qlin_status qlin_testing_qmv_chain_stalled(const void* x0, const qlin_link* links, int n_links,
                                           int bits, int group_size, qlin_dtype dtype,
                                           void* workspace, size_t workspace_bytes,
                                           int stalled_link, unsigned wait_limit_us,
                                           void* stream);

#ifdef __cplusplus
}
#endif

#endif /* QLIN_TESTING_H_ */
