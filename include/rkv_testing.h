/*
 * rkv_testing.h -- test hooks of the RocketKV library (not part of the method's interface).
 *
 * The kernels never spin without a bound: every wait on an mbarrier gives up after a time limit,
 * records RKV_DEV_WAIT_TIMEOUT in the workspace's status word, lets the copies it already issued
 * land, frees its tensor memory and returns, so that the CUDA context stays usable and the host
 * learns of the failure through rkv_check_status. This hook makes such a wait run out on purpose,
 * without any GPU fault, so that a test can check that path.
 */
#ifndef RKV_TESTING_H_
#define RKV_TESTING_H_

#include <stddef.h>
#include <stdint.h>

#include "rkv.h"

#ifdef __cplusplus
extern "C" {
#endif

/* rkv_snapkv_scores with every mbarrier wait of the score passes bounded by wait_limit_ns
 * (instead of 1 s) and with the first K tile of thread block 0's first pass-1 work item never
 * requested: the waits on that tile (the MMA issuer's, the epilogue's, and the producer's wait
 * for the stage to be released) run out after wait_limit_ns, block 0 records
 * RKV_DEV_WAIT_TIMEOUT and returns; every other block completes normally. Arguments, layouts and
 * errors as rkv_snapkv_scores; wait_limit_ns must be in [1000, 1e9]. The scores of the units
 * block 0 serves are not meaningful after such a call. */
rkv_status rkv_testing_scores_wait_timeout(const void* k, const int32_t* seq_lens,
                                           const void* q_win, int n, int n_kv, int gqa,
                                           int head_dim, int max_len, int window, float scale,
                                           float* scores_out, uint64_t wait_limit_ns, void* ws,
                                           size_t ws_bytes, void* stream);

/* Shared-memory layout of every later rkv_hybrid_decode call in this process, so that a test
 * can run each on the same inputs (the results do not depend on it; one CTA per (unit, KV head)
 * either way):
 *   0  automatic (the default): the wide layout -- every kept channel's summary row staged at
 *      once, every selected token's K / V rows staged per warp at once -- when there are no more
 *      (unit, KV head) pairs than SMs and it fits in shared memory, else the ordinary one;
 *   1  always the ordinary layout;
 *   2  the wide layout wherever it fits, whatever the number of units.
 * Returns RKV_ERR_INVALID_ARG (and changes nothing) for any other value. Not synchronised with
 * decode calls running on other host threads. */
rkv_status rkv_testing_decode_layout(int layout);

#ifdef __cplusplus
}
#endif

#endif /* RKV_TESTING_H_ */
