/*
 * gqa_attn_testing.h -- hooks of libgqa_attn.so that its own tests and
 * benchmark use: a self-test of the bounded device wait and per-kernel event
 * timing. They are exported by the same library but are NOT part of the
 * stable interface of gqa_attn.h: names, arguments and kernel numbering may
 * change with the kernels. Neither has a counterpart on the pages.
 */
#ifndef GQA_ATTN_TESTING_H
#define GQA_ATTN_TESTING_H

#include "gqa_attn.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Self-test of the bounded device wait (no counterpart on the pages): launches
 * one block that waits on an mbarrier nothing ever arrives at, with a limit of
 * limit_us microseconds (1..10^6). The kernel gives up, records the TIMEOUT
 * status bit and returns; a following gqa_attn_get_error() on the same
 * stream reports GQA_ERR_TIMEOUT (other streams' words are untouched). It faults, traps or hangs nothing.
 */
int gqa_attn_selftest_wait_timeout(int limit_us, void* stream);

/*
 * Per-kernel tracing (no counterpart on the pages; used to time each kernel
 * of a call live, e.g. for a roofline). gqa_attn_trace_arm() arms the calling
 * host thread: every kernel that gqa_attn_fwd / gqa_attn_bwd then launch from
 * this thread is bracketed by two CUDA events recorded on the call's stream.
 * gqa_attn_trace_collect() disarms, waits for the last recorded event, and
 * writes, for each kernel kind k (GQA_KERNEL_*), launches[k] and total_ms[k]
 * (arrays of GQA_KERNEL_COUNT entries, host memory, owned by the caller).
 * Events are created on first use on the device current at that time and
 * reused afterwards; no device memory is allocated.
 */
#define GQA_KERNEL_FWD 0
#define GQA_KERNEL_BWD_PREP 1
#define GQA_KERNEL_BWD_MAIN 2
#define GQA_KERNEL_BWD_CONVERT 3
#define GQA_KERNEL_DECODE_SPLIT 4
#define GQA_KERNEL_DECODE_COMBINE 5 /* no longer launched: the last chunk's CTA merges the partials */
#define GQA_KERNEL_BWD_DKDV 6 /* the deterministic backward's dK/dV kernel */
#define GQA_KERNEL_BWD_DQ 7   /* the deterministic backward's query-major dQ kernel */
#define GQA_KERNEL_ROPE 8     /* the rotary embedding's rotation pass */
#define GQA_KERNEL_FWD_COMBINE 9 /* the split forward's merge of its parts */
#define GQA_KERNEL_COUNT 10
int gqa_attn_trace_arm(void);
int gqa_attn_trace_collect(int* launches, double* total_ms);

#ifdef __cplusplus
}
#endif

#endif /* GQA_ATTN_TESTING_H */
