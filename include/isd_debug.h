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

#ifdef __cplusplus
}
#endif

#endif /* ISD_DEBUG_H_ */
