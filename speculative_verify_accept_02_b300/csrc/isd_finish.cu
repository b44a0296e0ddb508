// Per-sequence decisions of the ISD verify step and the per-row draws of the
// propose step, from the streaming pass's chunk partials ("Introspective
// Diffusion Language Models | Summary", §2 and §3.2).
//
// verify_finish_kernel, grid (C, nchunks), one CTA per (sequence, chunk):
//   decide  every CTA of sequence i merges the chunk partials of its rows into
//           log-partition values, forms ratio_k = min(1, p_k(x_k)/q_k(x_k)),
//           alpha_i and the accept prefix a_i (one warp ballot over k <= 32).
//           The decision is recomputed identically by each CTA; CTA 0 writes
//           it.
//   tail    a_i < L_i: CTA y sums the residual weights max(0, p_j - q_j) over
//           chunk y of the rejected rows (j = a_i + 1) — only that one row
//           pair is read again; a_i = L_i: CTA y reduces chunk y of the final
//           anchor row p_{L+1}.  Greedy rejections need no tail: the
//           correction is the argmax of p_j, known from the partials.
//   select  the last CTA of the sequence to finish its tail (atomic counter)
//           draws the token: chunk by inverse CDF over the chunk weights,
//           then an in-order scan of that one chunk.
// propose_sample_kernel, one CTA per qnew row: merge the row's partials, draw
//   by inverse CDF (argmax at T = 0), skipping sequences whose proposals would
//   be discarded.
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

// Residual weight of one id: max(0, p - q) with p, q the tempered softmaxes.
__device__ __forceinline__ float residual_weight(float xp, float xq, float Mp, float invSp, float Mq,
                                                 float invSq, float c2) {
    const float pv = ex2_approx((xp - Mp) * c2) * invSp;
    const float qv = ex2_approx((xq - Mq) * c2) * invSq;
    return fmaxf(0.0f, pv - qv);
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

__device__ __forceinline__ void block_softmax(float& M, float& S, float c2, float* sm, float* ss) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, M, o);
        const float s2 = __shfl_xor_sync(0xffffffffu, S, o);
        merge_softmax(M, S, m2, s2, c2);
    }
    __syncthreads();
    if (lane == 0) {
        sm[warp] = M;
        ss[warp] = S;
    }
    __syncthreads();
    M = -INFINITY;
    S = 0.0f;
    if (lane == 0) {
        for (int w = 0; w < kWarps; ++w) merge_softmax(M, S, sm[w], ss[w], c2);
    }
    M = __shfl_sync(0xffffffffu, M, 0);
    S = __shfl_sync(0xffffffffu, S, 0);
}

__device__ __forceinline__ void block_argmax(float& M, int& I, float* sm, int* si) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, M, o);
        const int i2 = __shfl_xor_sync(0xffffffffu, I, o);
        merge_argmax(M, I, m2, i2);
    }
    __syncthreads();
    if (lane == 0) {
        sm[warp] = M;
        si[warp] = I;
    }
    __syncthreads();
    M = -INFINITY;
    I = INT_MAX;
    for (int w = 0; w < kWarps; ++w) merge_argmax(M, I, sm[w], si[w]);
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
    float ratio[kMaxStride];
    float Mp[kMaxStride], Sp[kMaxStride], Mq[kMaxStride], Sq[kMaxStride];
    int amax[kMaxStride];
    float fs[2 * kWarps];
    int is[2 * kWarps];
    float alpha;
    int a;
    int last;
    int sel_chunk;
    float sel_t;
    float sel_M;
    int sel_mode;
    float w[kMaxChunkElems];
};

template <typename Elem>
__global__ void __launch_bounds__(kThreads) verify_finish_kernel(const VerifyFinishArgs a) {
    __shared__ Shared sh;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int i = blockIdx.x, y = blockIdx.y;
    const int NT = gridDim.y;

    pdl_wait();
    const SeqInfo s = seq_info(a.seq_offsets, a.temperature, i, a.total);
    const int err = *reinterpret_cast<const volatile int*>(a.err);
    bool ok = s.ok && err == 0;
    if (ok) {
        bool tok_ok = true;
        for (int k = tid; k < s.len; k += kThreads) {
            const int x = a.tokens[s.start + k];
            tok_ok = tok_ok && x >= 0 && x < a.vocab;
        }
        ok = __syncthreads_and(tok_ok);
    }
    if (!ok) {
        if (y == 0) {
            if (s.in_range) {
                for (int m = tid; m <= s.len; m += kThreads) a.out_tokens[s.start + i + m] = -1;
                for (int k = tid; k < s.len; k += kThreads) a.ratio[s.start + k] = NAN;
            }
            if (tid == 0) {
                a.accept_len[i] = err != 0 ? -2 : -1;
                a.alpha[i] = NAN;
            }
        }
        return;
    }
    const int L = s.len;
    const float T = s.T;
    const float c2 = T > 0.0f ? inv_temp_log2e(T) : 0.0f;

    // ---- decide -----------------------------------------------------------
    for (int k = warp; k < L; k += kWarps) {
        const int pos = s.start + k;
        const float2* pp = a.part + static_cast<size_t>(2 * pos) * a.nchunks;
        const float2* pq = pp + a.nchunks;
        if (T > 0.0f) {
            float M = -INFINITY, S = 0.0f, Mq = -INFINITY, Sq = 0.0f;
            for (int c = lane; c < a.nchunks; c += 32) {
                const float2 u = pp[c], v = pq[c];
                merge_softmax(M, S, u.x, u.y, c2);
                merge_softmax(Mq, Sq, v.x, v.y, c2);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float m2 = __shfl_xor_sync(0xffffffffu, M, o), s2 = __shfl_xor_sync(0xffffffffu, S, o);
                const float m3 = __shfl_xor_sync(0xffffffffu, Mq, o), s3 = __shfl_xor_sync(0xffffffffu, Sq, o);
                merge_softmax(M, S, m2, s2, c2);
                merge_softmax(Mq, Sq, m3, s3, c2);
            }
            if (lane == 0) {
                const float lp = (a.zx[2 * pos] - M) * c2 - log2f(S);
                const float lq = (a.zx[2 * pos + 1] - Mq) * c2 - log2f(Sq);
                sh.ratio[k] = lq == -INFINITY ? 1.0f : fminf(1.0f, exp2f(lp - lq));
                sh.Mp[k] = M;
                sh.Sp[k] = S;
                sh.Mq[k] = Mq;
                sh.Sq[k] = Sq;
            }
        } else {
            float M = -INFINITY;
            int I = INT_MAX;
            for (int c = lane; c < a.nchunks; c += 32) merge_argmax(M, I, pp[c].x, __float_as_int(pp[c].y));
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float m2 = __shfl_xor_sync(0xffffffffu, M, o);
                const int i2 = __shfl_xor_sync(0xffffffffu, I, o);
                merge_argmax(M, I, m2, i2);
            }
            if (lane == 0) {
                sh.amax[k] = I;
                sh.ratio[k] = a.tokens[pos] == I ? 1.0f : 0.0f;
            }
        }
    }
    __syncthreads();
    if (warp == 0) {
        const float r = lane < L ? sh.ratio[lane] : 0.0f;
        bool acc = false;
        if (lane < L)
            acc = T > 0.0f ? decision_uniform(a.seed, a.offset, i, lane + 1, kTagAccept) < r : r == 1.0f;
        const unsigned bits = __ballot_sync(0xffffffffu, acc);
        int na = bits == 0xffffffffu ? 32 : __ffs(~bits) - 1;
        na = min(na, L);
        const float total = warp_sum(r);
        if (lane == 0) {
            sh.a = na;
            sh.alpha = total / static_cast<float>(L);
        }
    }
    __syncthreads();
    const int na = sh.a;
    if (y == 0) {
        for (int k = tid; k < L; k += kThreads) a.ratio[s.start + k] = sh.ratio[k];
        for (int m = tid; m <= L; m += kThreads) {
            if (m < na) a.out_tokens[s.start + i + m] = a.tokens[s.start + m];
            else if (m > na) a.out_tokens[s.start + i + m] = -1;
        }
        if (tid == 0) {
            a.accept_len[i] = na;
            a.alpha[i] = sh.alpha;
            if (T == 0.0f && na < L) a.out_tokens[s.start + i + na] = sh.amax[na];
        }
    }
    if (T == 0.0f && na < L) return;

    // ---- tail: one chunk of the rows the draw needs ------------------------
    const bool bonus = na == L;
    const int e0 = y * a.chunk;
    const int n_el = min(a.chunk, a.vocab - e0);
    const char* prow = bonus ? a.p + static_cast<int64_t>(s.start + i + L) * a.ldp_bytes
                             : a.p + static_cast<int64_t>(s.start + i + na) * a.ldp_bytes;
    const char* qrow = a.q + static_cast<int64_t>(s.start + na) * a.ldq_bytes;
    float2 tp;
    if (bonus) {
        if (T > 0.0f) {
            float M = -INFINITY;
            for (int e = tid; e < n_el; e += kThreads) M = fmaxf(M, load_elem<Elem>(prow, e0 + e));
            float S = 0.0f;
            if (M != -INFINITY)
                for (int e = tid; e < n_el; e += kThreads) S += ex2_approx((load_elem<Elem>(prow, e0 + e) - M) * c2);
            block_softmax(M, S, c2, sh.fs, sh.fs + kWarps);
            tp = make_float2(M, S);
        } else {
            float M = -INFINITY;
            int I = INT_MAX;
            for (int e = tid; e < n_el; e += kThreads) merge_argmax(M, I, load_elem<Elem>(prow, e0 + e), e0 + e);
            block_argmax(M, I, sh.fs, sh.is);
            tp = make_float2(M, __int_as_float(I));
        }
    } else {
        const float Mp = sh.Mp[na], invSp = 1.0f / sh.Sp[na];
        const float Mq = sh.Mq[na], invSq = 1.0f / sh.Sq[na];
        float acc = 0.0f;
        for (int e = tid; e < n_el; e += kThreads)
            acc += residual_weight(load_elem<Elem>(prow, e0 + e), load_elem<Elem>(qrow, e0 + e), Mp, invSp,
                                   Mq, invSq, c2);
        tp = make_float2(block_sum(acc, sh.fs), 0.0f);
    }
    if (tid == 0) {
        a.tail_part[static_cast<size_t>(i) * NT + y] = tp;
        __threadfence();
        sh.last = atomicAdd(a.tail_count + i, 1) == NT - 1;
    }
    __syncthreads();
    if (!sh.last) return;
    __threadfence();

    // ---- select: the last CTA of the sequence draws the token -------------
    const float2* tparts = a.tail_part + static_cast<size_t>(i) * NT;
    if (tid == 0) {
        int mode = bonus ? 1 : 0;  // 0 residual, 1 softmax of p_{L+1}, 2 softmax of p_j
        float M = -INFINITY, S = 0.0f;
        int chosen = -1;
        float tloc = 0.0f;
        if (bonus && T == 0.0f) {
            int I = INT_MAX;
            for (int c = 0; c < NT; ++c) {
                const float2 v = __ldcg(tparts + c);
                merge_argmax(M, I, v.x, __float_as_int(v.y));
            }
            a.out_tokens[s.start + i + L] = I;
            mode = -1;
        } else {
            const float2* wparts = tparts;
            if (!bonus) {
                for (int c = 0; c < NT; ++c) S += __ldcg(tparts + c).x;
                if (!(S > 0.0f)) {
                    // All residual weights rounded to zero: draw from p_j.
                    mode = 2;
                    wparts = a.part + static_cast<size_t>(2 * (s.start + na)) * a.nchunks;
                }
            }
            if (mode != 0) {
                for (int c = 0; c < NT; ++c) {
                    const float2 v = __ldcg(wparts + c);
                    merge_softmax(M, S, v.x, v.y, c2);
                }
            }
            const float u = bonus ? decision_uniform(a.seed, a.offset, i, L + 1, kTagBonus)
                                  : decision_uniform(a.seed, a.offset, i, na + 1, kTagCorrect);
            // Chunk weights in one scale, then the chunk holding t = u * S.
            float total = 0.0f;
            for (int c = 0; c < NT; ++c) {
                const float2 v = __ldcg(wparts + c);
                total += mode == 0 ? v.x : (v.x == -INFINITY ? 0.0f : v.y * exp2f((v.x - M) * c2));
            }
            const float t = u * total;
            float cum = 0.0f;
            int last_pos = -1;
            for (int c = 0; c < NT; ++c) {
                const float2 v = __ldcg(wparts + c);
                const float wc = mode == 0 ? v.x : (v.x == -INFINITY ? 0.0f : v.y * exp2f((v.x - M) * c2));
                if (wc > 0.0f) last_pos = c;
                if (chosen < 0 && cum + wc > t) {
                    chosen = c;
                    tloc = t - cum;
                }
                cum += wc;
            }
            if (chosen < 0) {
                chosen = last_pos;
                tloc = INFINITY;
            }
            if (chosen < 0) chosen = 0;  // no positive weight at all (non-finite logits)
        }
        sh.sel_mode = mode;
        sh.sel_chunk = chosen;
        sh.sel_t = tloc;
        sh.sel_M = M;
    }
    __syncthreads();
    const int mode = sh.sel_mode;
    if (mode < 0) return;
    const int cs = sh.sel_chunk;
    const int c0 = cs * a.chunk;
    const int cn = min(a.chunk, a.vocab - c0);
    if (mode == 0) {
        const float Mp = sh.Mp[na], invSp = 1.0f / sh.Sp[na];
        const float Mq = sh.Mq[na], invSq = 1.0f / sh.Sq[na];
        for (int e = tid; e < cn; e += kThreads)
            sh.w[e] = residual_weight(load_elem<Elem>(prow, c0 + e), load_elem<Elem>(qrow, c0 + e), Mp, invSp,
                                      Mq, invSq, c2);
    } else {
        const float M = sh.sel_M;
        for (int e = tid; e < cn; e += kThreads) sh.w[e] = ex2_approx((load_elem<Elem>(prow, c0 + e) - M) * c2);
    }
    __syncthreads();
    const int v = scan_chunk(sh.w, cn, sh.sel_t, sh.fs, sh.is);
    if (tid == 0) a.out_tokens[s.start + i + na] = c0 + v;
}

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

cudaError_t launch_verify_finish(const VerifyFinishArgs& a, int elem_bytes, cudaStream_t stream) {
    const dim3 grid(a.num_seqs, a.nchunks);
    return elem_bytes == 2 ? launch_pdl(verify_finish_kernel<__nv_bfloat16>, grid, dim3(kThreads), stream, a)
                           : launch_pdl(verify_finish_kernel<float>, grid, dim3(kThreads), stream, a);
}

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
