/*
 * dsa_testhooks.h -- the one extra entry point of the TEST build of the library,
 * libdsa_testhooks.so (the same sources compiled with -DDSA_TEST_HOOKS).  The product library
 * libdsa.so does not export it.  The pages have no counterpart: this exists so that the
 * failure handling of the kernels can be exercised without faulting or hanging a GPU.
 *
 * In the test build every bounded device-side wait gives up after 20 ms (1 s in the product).
 *
 * dsa_test_inject_stall(kernel): from the next launch on, the single MMA-issuing thread of the
 * first CTA of the chosen kernel (1: the indexer, dsa_li_topk; 2: sparse attention,
 * dsa_sfa_decode / dsa_sfa_prefill; 0: none) first waits on an mbarrier that no thread ever
 * arrives on.  That wait runs out, the CTA raises its abort flag, the kernel stores
 * DSA_ERR_TIMEOUT into *status, the other roles of the CTA (and of its cluster) leave their
 * loops through their own bounded waits, every issued copy is drained, tensor memory is
 * freed, and the launch completes: the next call on the same context works.  The output of the
 * stalled launch is unspecified.  Host-side state, not thread-safe; a test setting.
 */
#ifndef DSA_TESTHOOKS_H
#define DSA_TESTHOOKS_H

#ifdef __cplusplus
extern "C" {
#endif

void dsa_test_inject_stall(int kernel);

#ifdef __cplusplus
}
#endif

#endif /* DSA_TESTHOOKS_H */
