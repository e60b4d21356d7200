/*
 * qlin_testing.h -- entry points of libqlin that exist only for the library's
 * own tests: to reach failure paths without faulting or hanging a GPU, and to
 * check host-side launch choices without one.  They have no counterpart on
 * the pages the method comes from, and no product code calls them.
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

/*
 * The split of K that qlin_qmv (and qlin_linear's qmv path) would use for an
 * N x K matrix of `bits`-bit codes on a device with `sm_count` SMs: the
 * number of CTAs (a thread-block cluster) that share each row block, each
 * taking an equal share of the row's k-tiles (1: no split).  Host logic only;
 * touches no device.  Honours the QLIN_QMV_SPLIT and QLIN_QMV_R tuning
 * variables as the launcher does.  Returns -1 for arguments qlin_qmv would
 * reject (bits not 4 or 8, K not a positive multiple of 64, N < 1) or
 * sm_count < 1.
 */
int qlin_testing_qmv_split(int64_t N, int64_t K, int bits, int sm_count);

#ifdef __cplusplus
}
#endif

#endif /* QLIN_TESTING_H_ */
