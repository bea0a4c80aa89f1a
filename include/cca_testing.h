/*
 * cca_testing.h - test hooks of libcca.so.  Not for production callers.
 *
 * The first two exercise the bounded-wait path of the bf16 attention kernel without
 * faulting or hanging the GPU: every mbarrier wait in that kernel gives up
 * after a time limit, raises a CTA-wide abort flag, drains the copies and
 * tensor-core operations it already issued, frees its tensor memory and
 * writes CCA_ERR_TIMEOUT into the caller's dev_status word.
 *
 * All settings are process-wide and apply to launches made after the call;
 * they are not thread-safe with respect to concurrent launches.
 */
#ifndef CCA_TESTING_H_
#define CCA_TESTING_H_

#ifdef __cplusplus
extern "C" {
#endif

/* Per-wait time limit in nanoseconds for later bf16 tensor-core launches,
 * forward and backward (default 1e9, i.e. one second). */
void cca_test_set_wait_limit_ns(unsigned long long ns);

/* on != 0: later bf16 attention launches never load the query tile, so the
 * tensor-core issuer's first wait runs out and the kernel reports a time-out;
 * the tensor-core backward kernels issue no copies at all, so their first wait
 * runs out the same way.  on == 0 restores normal operation. */
void cca_test_skip_q_load(int on);

/* Which decode path later cca_decode_fwd / cca_decode_fwd_noalloc calls take:
 * 1 the split kernel + merge kernel through the workspace, 2 the single
 * launch whose splits merge inside a thread-block cluster (where a cluster of
 * two or more splits fits), anything else the automatic choice. */
void cca_test_decode_path(int path);

#ifdef __cplusplus
}
#endif

#endif /* CCA_TESTING_H_ */
