// Per-row draws of the propose step from the streaming pass's chunk
// partials ("Introspective Diffusion Language Models | Summary", §3.2: the
// mask positions of a forward give the next stride's proposals).
//
// propose_sample_kernel, one CTA per qnew row: merge the row's partials, draw
//   by inverse CDF (argmax at T = 0), skipping sequences whose proposals would
//   be discarded.  The chunk holding the target comes from the partials; only
//   that chunk is read again and scanned in vocabulary order.
#include <climits>

#include "isd_device.cuh"
#include "isd_internal.h"

namespace isd {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxChunkElems = kStageBytes / 2;  // bf16 chunk bound (fp32: half)

template <typename Elem>
__device__ __forceinline__ float load_elem(const char* row, int e) {
    if constexpr (sizeof(Elem) == 2)
        return __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(row)[e]) << 16);
    else
        return reinterpret_cast<const float*>(row)[e];
}

__device__ __forceinline__ float block_sum(float v, float* scratch) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    v = warp_sum(v);
    __syncthreads();
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    float t = lane < kWarps ? scratch[lane] : 0.0f;
    return warp_sum(t);
}

// In-order inverse-CDF scan of one chunk whose weights are in w[0..n): the
// smallest e whose running sum exceeds t; if rounding leaves none, the last e
// with positive weight.  Returns the chunk-relative index (all threads).
__device__ int scan_chunk(const float* w, int n, float t, float* fscratch, int* iscratch) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int seg = (n + kThreads - 1) / kThreads;
    const int b = min(n, tid * seg), e = min(n, b + seg);
    float own = 0.0f;
    for (int k = b; k < e; ++k) own += w[k];
    // Inclusive scan of the per-thread sums in thread order.
    float incl = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float x = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += x;
    }
    __syncthreads();
    if (lane == 31) fscratch[warp] = incl;
    __syncthreads();
    float before_warp = 0.0f;
    for (int k = 0; k < warp; ++k) before_warp += fscratch[k];
    incl += before_warp;
    const float excl = incl - own;
    int cand = INT_MAX;
    if (incl > t && e > b) {
        float c = excl;
        for (int k = b; k < e; ++k) {
            c += w[k];
            if (c > t) {
                cand = k;
                break;
            }
        }
    }
    int last_pos = -1;
    for (int k = b; k < e; ++k)
        if (w[k] > 0.0f) last_pos = k;
    cand = warp_min_int(cand);
    last_pos = warp_max_int(last_pos);
    __syncthreads();
    if (lane == 0) {
        iscratch[warp] = cand;
        iscratch[kWarps + warp] = last_pos;
    }
    __syncthreads();
    int best = INT_MAX, lastp = -1;
    for (int k = 0; k < kWarps; ++k) {
        best = min(best, iscratch[k]);
        lastp = max(lastp, iscratch[kWarps + k]);
    }
    return best != INT_MAX ? best : lastp;
}

struct Shared {
    float fs[2 * kWarps];
    int is[2 * kWarps];
    int sel_chunk;
    float sel_t;
    float sel_M;
    float w[kMaxChunkElems];
};

template <typename Elem>
__global__ void __launch_bounds__(kThreads) propose_sample_kernel(const ProposeSampleArgs a) {
    __shared__ Shared sh;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b = blockIdx.x;
    pdl_wait();
    const int err = *reinterpret_cast<const volatile int*>(a.err);
    if (b < a.num_seqs && tid == 0) {
        const SeqInfo si = seq_info(a.seq_offsets, a.temperature, b, a.total);
        bool ok = si.ok && err == 0;
        if (ok && a.accept_len != nullptr) ok = a.accept_len[b] == si.len;
        a.valid[b] = ok ? 1 : 0;
    }
    if (b >= a.total) return;
    const int r = b;
    const int i = seq_of_position(a.seq_offsets, a.num_seqs, r);
    const SeqInfo s = seq_info(a.seq_offsets, a.temperature, i, a.total);
    bool ok = s.ok && err == 0 && r >= s.start && r < s.start + s.len;
    if (ok && a.accept_len != nullptr) ok = a.accept_len[i] == s.len;
    if (!ok) {
        if (tid == 0) a.proposals[r] = -1;
        return;
    }
    const int m = r - s.start + 1;
    const float T = s.T;
    const float c2 = T > 0.0f ? inv_temp_log2e(T) : 0.0f;
    const float2* pr = a.part + static_cast<size_t>(r) * a.nchunks;
    if (T == 0.0f) {
        if (warp == 0) {
            float M = -INFINITY;
            int I = INT_MAX;
            for (int c = lane; c < a.nchunks; c += 32) merge_argmax(M, I, pr[c].x, __float_as_int(pr[c].y));
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float m2 = __shfl_xor_sync(0xffffffffu, M, o);
                const int i2 = __shfl_xor_sync(0xffffffffu, I, o);
                merge_argmax(M, I, m2, i2);
            }
            if (lane == 0) a.proposals[r] = I;
        }
        return;
    }
    if (tid == 0) {
        float M = -INFINITY, S = 0.0f;
        for (int c = 0; c < a.nchunks; ++c) merge_softmax(M, S, pr[c].x, pr[c].y, c2);
        float total = 0.0f;
        for (int c = 0; c < a.nchunks; ++c)
            total += pr[c].x == -INFINITY ? 0.0f : pr[c].y * exp2f((pr[c].x - M) * c2);
        const float u = decision_uniform(a.seed, a.offset, i, m, kTagPropose);
        const float t = u * total;
        float cum = 0.0f;
        int chosen = -1, last_pos = -1;
        float tloc = INFINITY;
        for (int c = 0; c < a.nchunks; ++c) {
            const float wc = pr[c].x == -INFINITY ? 0.0f : pr[c].y * exp2f((pr[c].x - M) * c2);
            if (wc > 0.0f) last_pos = c;
            if (chosen < 0 && cum + wc > t) {
                chosen = c;
                tloc = t - cum;
            }
            cum += wc;
        }
        if (chosen < 0) chosen = last_pos;
        if (chosen < 0) chosen = 0;  // no positive weight at all (non-finite logits)
        sh.sel_chunk = chosen;
        sh.sel_t = tloc;
        sh.sel_M = M;
    }
    __syncthreads();
    const char* row = a.rows + static_cast<int64_t>(r) * a.ld_bytes;
    const int c0 = sh.sel_chunk * a.chunk;
    const int cn = min(a.chunk, a.vocab - c0);
    const float M = sh.sel_M;
    for (int e = tid; e < cn; e += kThreads) sh.w[e] = ex2_approx((load_elem<Elem>(row, c0 + e) - M) * c2);
    __syncthreads();
    const int v = scan_chunk(sh.w, cn, sh.sel_t, sh.fs, sh.is);
    if (tid == 0) a.proposals[r] = c0 + v;
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

template <typename Kernel, typename Args>
cudaError_t launch_pdl(Kernel kernel, dim3 grid, dim3 block, cudaStream_t stream, const Args& args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args);
}

}  // namespace

cudaError_t launch_propose_sample(const ProposeSampleArgs& a, int elem_bytes, cudaStream_t stream) {
    const dim3 grid(max(a.total, a.num_seqs));
    return elem_bytes == 2 ? launch_pdl(propose_sample_kernel<__nv_bfloat16>, grid, dim3(kThreads), stream, a)
                           : launch_pdl(propose_sample_kernel<float>, grid, dim3(kThreads), stream, a);
}

cudaError_t launch_alpha(const float* ratio, const int32_t* seq_offsets, int num_seqs, int total,
                         float* alpha_per_seq, float* alpha_mean, cudaStream_t stream) {
    alpha_kernel<<<1, kThreads, 0, stream>>>(ratio, seq_offsets, num_seqs, total, alpha_per_seq, alpha_mean);
    return cudaGetLastError();
}

}  // namespace isd
