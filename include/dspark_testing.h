/*
 * dspark_testing.h -- diagnostic and measurement entry points of libdspark.
 *
 * These calls have no counterpart in the DSpark paper and are not part of the
 * method's interface (include/dspark.h). The library exports them for its own
 * tests and benchmark: a self-test of the bounded device-side waits, and
 * variants of dspark_verify and dspark_draft_markov that record caller-owned
 * CUDA events between their kernels. Conventions are those of dspark.h.
 */
#ifndef DSPARK_TESTING_H
#define DSPARK_TESTING_H

#include "dspark.h"

#ifdef __cplusplus
extern "C" {
#endif

struct CUevent_st; /* cudaEvent_t / CUevent */

/*
 * dspark_wait_selftest -- a diagnostic of the bounded waits (no counterpart in
 * the paper). Every wait in the library gives up after about a second of the
 * device's global timer, writes DSPARK_ERR_TIMEOUT to the status word and lets
 * its kernel return, so that a lost completion never hangs the GPU. This call
 * runs one such wait on a condition that never comes true, in one CTA:
 *   which 0  the ring waits of the pipelines: an mbarrier that no copy and no
 *            thread completes;
 *   which 1  the drafter's barrier among the CTAs of a request tile: two CTAs
 *            expected in a grid of one;
 *            sync_words = 8 bytes of caller device memory, zeroed before the
 *            call (left holding one arrival).
 * The kernel records DSPARK_ERR_TIMEOUT in *device_status (if it holds
 * DSPARK_OK) after about a second and returns; later calls on the stream run
 * normally. Host errors: which not 0 or 1, device_status NULL, or (which 1)
 * sync_words NULL or not 8-byte aligned -> DSPARK_ERR_INVALID_ARG.
 */
int dspark_wait_selftest(int32_t which, void* sync_words, int32_t* device_status,
                         struct CUstream_st* stream);

/*
 * dspark_verify_timed -- dspark_verify with per-pass timing events (a
 * measurement aid; no counterpart in the paper).
 *
 * Does exactly the work of dspark_verify and also records, on `stream`:
 *   events[0] before the planning pass (k_plan),
 *   events[1] before the streaming pass (k_rowstats),
 *   events[2] before the decision pass (k_decide: ratio tests, residual sums
 *             and the draw),
 *   events[3] after it.
 * cudaEventElapsedTime(events[i], events[i+1]), after the caller's own
 * synchronisation, gives the duration of pass i. events points to 4 events
 * the caller created with timing enabled (cudaEventCreate) and still owns.
 * Recording between the passes stops a pass's launch from overlapping the end
 * of the previous one, so the three intervals add up to slightly more than a
 * dspark_verify call takes.
 *
 * Arguments, outputs and error behaviour are those of dspark_verify; a NULL
 * events pointer or event is DSPARK_ERR_INVALID_ARG.
 */
int dspark_verify_timed(const void* target_logits, const void* draft_logits,
                        const int32_t* draft_tokens, const int32_t* verify_len,
                        const float* uniforms, float temperature, int32_t dtype,
                        int32_t B, int32_t gamma, int32_t V,
                        const int64_t* target_row_off, const int64_t* draft_row_off,
                        int32_t* accepted_len, int32_t* emitted_tokens,
                        float* probs_out, uint32_t* near_tie_count,
                        int32_t* device_status, void* workspace,
                        size_t workspace_bytes, struct CUstream_st* stream,
                        struct CUevent_st** events);

/*
 * dspark_draft_markov_timed -- dspark_draft_markov with timing events (a
 * measurement aid; no counterpart in the paper). Records events[0] before the
 * first gather, events[1] after it, and for k = 0..gamma-1 events[2+2k] after
 * position k's tensor-core kernel (k_draft_step) and events[3+2k] after its
 * draw (k_draft_pick): 2*gamma + 2 events created by the caller with timing
 * enabled. The recordings keep consecutive kernels from overlapping, so the
 * intervals add up to a little more than an untimed call. A NULL events
 * pointer or event is DSPARK_ERR_INVALID_ARG.
 */
int dspark_draft_markov_timed(const void* base_logits, const void* w1, const void* w2t,
                              const int32_t* anchors, const float* uniforms,
                              float temperature, int32_t B, int32_t gamma, int64_t V,
                              int32_t r, void* draft_logits, int32_t* draft_tokens,
                              int32_t* device_status, void* workspace,
                              size_t workspace_bytes, struct CUstream_st* stream,
                              struct CUevent_st** events);

#ifdef __cplusplus
}
#endif

#endif /* DSPARK_TESTING_H */
