/*
 * isd_debug.h — C ABI of libisd's check entry points: calls that expose one
 * building block of the step so that it can be compared with an independent
 * implementation, bit for bit.  They are not part of the step.
 *
 * The conventions of include/isd.h hold (device pointers owned by the
 * caller, one launch on `stream`, nothing allocated or synchronised).
 */
#ifndef ISD_DEBUG_H_
#define ISD_DEBUG_H_

#include "isd.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * isd_decision_uniforms — the uniforms the kernels draw for their decisions
 * (include/isd.h, "Random numbers"): out[j] = u(seed, offset, seq_j, pos_j,
 * tag_j) for j < n, where counters[3 j .. 3 j + 2] = (seq_j, pos_j, tag_j):
 * Philox4x64-10 with key (seed, 0) and counter (offset, seq_j, pos_j,
 * tag_j), the top 24 bits of output word 0 times 2^-24.
 *
 * counters [3 n] uint64 (device), out [n] float (device).  n = 0 launches
 * nothing; n < 0 or a NULL pointer with n > 0 returns ISD_ERR_INVALID_ARG.
 */
ISD_API isd_status isd_decision_uniforms(uint64_t seed, uint64_t offset, const uint64_t* counters, int n,
                                         float* out, void* stream);

/*
 * isd_debug_verify_stall — isd_verify_propose with one sequence's decision
 * held back, to test the verify kernel's bounded waits without a GPU fault
 * (failure detection).  The decision of sequence `stall_seq` writes its
 * outputs and reserves the queue slot of its correction or bonus draw but
 * never publishes that draw's descriptor, so the worker warps holding the
 * draw's piece tickets poll for it until their bound on waits for other
 * CTAs' work runs out: `wait_ns` nanoseconds of the global timer instead of
 * the usual 4 s.  The hook takes effect on a sequence with T > 0 (a T = 0
 * sequence that does not accept its whole stride has no draw to hold back).
 * The call then ends as a timeout does: the workspace's
 * error word is set, every accept_len reads -2 and every valid 0, and the
 * workspace must be zero-filled again before its next use (include/isd.h,
 * Workspace).  Only waits on other CTAs' work can run out this way: every
 * bulk copy of the kernel has landed before any CTA exits.
 *
 * stall_seq in [-1, num_seqs) (-1: no stall, an ordinary call with the
 * shorter bound); wait_ns in [10^5, 4 10^9] (ISD_ERR_INVALID_ARG
 * otherwise).  A bound far below the call's own duration can run out on an
 * ordinary call too.  Every other argument as isd_verify_propose.
 */
ISD_API isd_status isd_debug_verify_stall(const void* p_logits, int64_t ld_p, const void* q_logits, int64_t ld_q,
                                          isd_dtype dtype, int vocab, const int32_t* tokens,
                                          const int32_t* seq_offsets, int num_seqs, int total_positions,
                                          const float* temperature, uint64_t seed, uint64_t offset,
                                          int32_t* accept_len, int32_t* out_tokens, float* ratio, float* alpha,
                                          const void* qnew_logits, int64_t ld_qnew, int32_t* proposals,
                                          uint8_t* valid, void* workspace, size_t workspace_bytes, int stall_seq,
                                          uint64_t wait_ns, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* ISD_DEBUG_H_ */
