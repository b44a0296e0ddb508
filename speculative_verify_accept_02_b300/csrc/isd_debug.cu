// Check entry points (include/isd_debug.h): the building blocks of the step,
// exposed one at a time so that they can be compared bit for bit with an
// independent implementation.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/isd_debug.h"
#include "isd_device.cuh"
#include "isd_internal.h"

namespace isd {
namespace {

constexpr int kThreads = 256;

// One uniform per counter triple, with the same device function the
// decision, selection and proposal code calls.
__global__ void __launch_bounds__(kThreads) uniforms_kernel(uint64_t seed, uint64_t offset, const uint64_t* ctr,
                                                          int n, float* out) {
    for (long long j = blockIdx.x * static_cast<long long>(kThreads) + threadIdx.x; j < n;
         j += static_cast<long long>(gridDim.x) * kThreads)
        out[j] = decision_uniform(seed, offset, ctr[3 * j], ctr[3 * j + 1], ctr[3 * j + 2]);
}

}  // namespace
}  // namespace isd

extern "C" isd_status isd_decision_uniforms(uint64_t seed, uint64_t offset, const uint64_t* counters, int n,
                                            float* out, void* stream) {
    if (n < 0 || (n > 0 && (!counters || !out))) return ISD_ERR_INVALID_ARG;
    if (n == 0) return ISD_OK;
    const int blocks = (n + isd::kThreads - 1) / isd::kThreads;
    const int grid = blocks < 1024 ? blocks : 1024;
    isd::uniforms_kernel<<<grid, isd::kThreads, 0, static_cast<cudaStream_t>(stream)>>>(seed, offset, counters, n,
                                                                                        out);
    return cudaGetLastError() == cudaSuccess ? ISD_OK : ISD_ERR_CUDA;
}

extern "C" isd_status isd_debug_verify_stall(const void* p_logits, int64_t ld_p, const void* q_logits, int64_t ld_q,
                                             isd_dtype dtype, int vocab, const int32_t* tokens,
                                             const int32_t* seq_offsets, int num_seqs, int total_positions,
                                             const float* temperature, uint64_t seed, uint64_t offset,
                                             int32_t* accept_len, int32_t* out_tokens, float* ratio, float* alpha,
                                             const void* qnew_logits, int64_t ld_qnew, int32_t* proposals,
                                             uint8_t* valid, void* workspace, size_t workspace_bytes,
                                             int stall_seq, uint64_t wait_ns, void* stream) {
    if (stall_seq < -1 || stall_seq >= num_seqs) return ISD_ERR_INVALID_ARG;
    if (wait_ns < 100000ull || wait_ns > isd::kVerifyWaitNs) return ISD_ERR_INVALID_ARG;
    isd::VerifyOptions o;
    o.fused = true;
    o.qnew = qnew_logits;
    o.ld_qnew = ld_qnew;
    o.proposals = proposals;
    o.valid = valid;
    o.wait_ns = wait_ns;
    o.stall_seq = stall_seq;
    return isd::verify_run(p_logits, ld_p, q_logits, ld_q, dtype, vocab, tokens, seq_offsets, num_seqs,
                           total_positions, temperature, seed, offset, accept_len, out_tokens, ratio, alpha, o,
                           workspace, workspace_bytes, stream);
}
