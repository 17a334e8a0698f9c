/*
 * kda_testing.h -- test hooks of libkda.  NOT for production use.
 *
 * The course pages have no counterpart to these calls.  They exist so that
 * the library's own tests can (a) run the tensor-core prefill under each of
 * its launch plans, which must give bit-identical results, and (b) drive a
 * bounded device-side wait to expiry and check that the failure is reported
 * as KDA_ERR_TIMEOUT by kda_prefill_check while the context stays usable.
 *
 * Both hooks set process-wide state that every later kda_prefill_chunked
 * call on any thread reads at launch time; a test must restore the defaults
 * (plan -1, fault KDA_TESTING_FAULT_NONE with wait limit 0) when it is done.
 */
#ifndef KDA_TESTING_H_
#define KDA_TESTING_H_

#include "kda.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Launch plans of the tensor-core prefill (bf16, d = 128, chunk 64). */
#define KDA_TESTING_PLAN_AUTO (-1)  /* the library chooses (the default) */
#define KDA_TESTING_PLAN_THREE 0    /* preparation, then the state pass, which also forms the outputs (with the
                                       gated output normalisation fused: state pass, then output pass) */
#define KDA_TESTING_PLAN_CHAIN 2    /* preparation, then one cooperative launch of the state chains with the
                                       output units alongside; falls back to THREE where it cannot run */
#define KDA_TESTING_PLAN_PIPE 3     /* one cooperative launch: state chains (32 or 64 columns) beside groups that
                                       prepare the records in chunk order and form the outputs behind the
                                       chains; falls back to THREE where it cannot run */

/* Forces a launch plan for later calls.  KDA_ERR_INVALID_ARG for an unknown plan. */
KDA_API kda_status kda_testing_set_plan(int32_t plan);

/* Faults for tests of the failure path. */
#define KDA_TESTING_FAULT_NONE 0        /* the default */
#define KDA_TESTING_FAULT_NO_PUBLISH 1  /* chain and pipe plans: the state chains publish none of their state
                                           images, so the output units' bounded waits on them run out */
#define KDA_TESTING_FAULT_CHUNK_TABLE 2 /* bounds-checking build (libkda_debug.so) only: the chunk table claims
                                           1000 chunks more than exist, which the kernels' bounds checks must
                                           catch (KDA_ERR_BOUNDS); the release build ignores this fault */

/*
 * Injects `fault` into later calls and bounds the device-side waits on
 * another CTA's publication flag by `wait_limit_ns` nanoseconds (0 keeps the
 * default of two seconds).  KDA_ERR_INVALID_ARG for an unknown fault or a
 * negative limit.
 */
KDA_API kda_status kda_testing_set_fault(int32_t fault, int64_t wait_limit_ns);

#ifdef __cplusplus
}
#endif

#endif /* KDA_TESTING_H_ */
