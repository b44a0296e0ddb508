// Introspective acceptance rate from per-position ratios ("Introspective
// Diffusion Language Models | Summary", §2): the mean ratio of each
// sequence's stride and the mean over the batch.
#include "isd_device.cuh"
#include "isd_internal.h"

namespace isd {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ float block_sum(float v, float* scratch) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    v = warp_sum(v);
    __syncthreads();
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    float t = lane < kWarps ? scratch[lane] : 0.0f;
    return warp_sum(t);
}

__global__ void __launch_bounds__(kThreads) alpha_kernel(const float* ratio, const int32_t* offs, int C,
                                                         int total, float* per, float* mean) {
    __shared__ float scratch[kWarps];
    float acc = 0.0f;
    for (int i = threadIdx.x; i < C; i += kThreads) {
        const int b = offs[i], e = offs[i + 1];
        float v = NAN;
        if (b >= 0 && e <= total && e > b) {
            float s = 0.0f;
            for (int k = b; k < e; ++k) s += ratio[k];
            v = s / static_cast<float>(e - b);
        }
        per[i] = v;
        acc += v;
    }
    const float t = block_sum(acc, scratch);
    if (threadIdx.x == 0) *mean = t / static_cast<float>(C);
}

}  // namespace

cudaError_t launch_alpha(const float* ratio, const int32_t* seq_offsets, int num_seqs, int total,
                         float* alpha_per_seq, float* alpha_mean, cudaStream_t stream) {
    alpha_kernel<<<1, kThreads, 0, stream>>>(ratio, seq_offsets, num_seqs, total, alpha_per_seq, alpha_mean);
    return cudaGetLastError();
}

}  // namespace isd
