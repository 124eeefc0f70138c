/*
 * mla_test.h — test hooks of the MLA decode library (not part of a decode step).
 *
 * The pages describe no failure handling; this entry exists so that a test can
 * drive the decode kernel's abort path for real without breaking anything: every
 * wait inside mla_decode_fwd is bounded, and when one runs out the kernel records
 * MLA_ERR_TIMEOUT in the status word, tells the peer CTA of its SM pair to stop,
 * waits (with the long limit) for the copies and tensor-core work it already
 * started, frees its tensor memory and returns, leaving the stream usable.
 */
#ifndef MLA_TEST_H_
#define MLA_TEST_H_

#include "mla.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * mla_test_decode_stalled — mla_decode_fwd (bf16 cache only, same arguments and
 * schedule) in which the score CTA of every SM pair issues none of its loads, so the
 * waits of the roles that consume them run out, and every wait that an abort can end
 * has the limit `wait_ns` instead of 2 s.
 *   status   device int32, required (the caller zeroes it); receives MLA_ERR_TIMEOUT
 *   wait_ns  1000 .. 2e9
 * Returns MLA_OK once the launch is queued (or the host-side errors of
 * mla_decode_fwd; MLA_ERR_INVALID_ARG for an e4m3 cache, a NULL status or a
 * limit out of range). o_part / lse_part are left undefined.
 */
MLA_API mla_status mla_test_decode_stalled(const void* q_lat, const mla_cache* cache,
                                           const int32_t* seq_lens, int B, int n_h,
                                           int max_seq_len, float softmax_scale,
                                           int num_splits, float* o_part, float* lse_part,
                                           int32_t* status, uint64_t wait_ns,
                                           cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MLA_TEST_H_ */
