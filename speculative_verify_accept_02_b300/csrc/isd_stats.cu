// Streaming pass over vocabulary rows: the HBM-bound part of the ISD
// verify-and-propose step ("Introspective Diffusion Language Models |
// Summary", §3.3: the verification uses an online softmax).
//
// Every (row, chunk) item is read once from HBM by a 1-D bulk copy into a
// shared-memory stage and reduced by eight consumer warps to one partial:
//   T > 0: (m, s) with m the chunk's largest logit and
//          s = sum exp2((x - m) * log2(e) / T), carried in fp32;
//   T = 0: (m, lowest id holding m), exact.
// Verified rows also record the logit of their proposed token.
//
// Persistent grid (2 CTAs per SM), items dealt round-robin; one producer
// thread keeps kStages bulk copies in flight per CTA, the consumer warps
// release a stage as soon as its data is in registers.
#include <climits>

#include "isd_device.cuh"
#include "isd_internal.h"

namespace isd {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kStatsThreads = kConsumerThreads + 32;  // + one producer warp
constexpr int kStages = 4;
constexpr int kVecPerThread = kStageBytes / 16 / kConsumerThreads;
static_assert(kVecPerThread * 16 * kConsumerThreads == kStageBytes, "stage split");

struct ItemDesc {
    const char* tail_src;  // global address of the first element not in shared memory
    int slot;
    int chunk;
    int n_smem;            // chunk elements held in shared memory
    int skip;              // elements in shared memory before the chunk start
    int n_tail;            // chunk elements read from global memory
    int tma_bytes;         // bytes of the bulk copy
    int gather;            // chunk-relative index of the proposed token, or -1
    float c2;              // log2(e)/T, or 0 for an argmax row
    int end;               // 1: no more items
};

struct StatsSmem {
    alignas(128) unsigned char stage[kStages][kStageBytes];
    uint64_t full[kStages];
    uint64_t empty[kStages];
    ItemDesc desc[kStages];
    float2 red[2][kConsumerWarps];
    int redi[2][kConsumerWarps];
    int abort;
};

template <typename Elem>
struct Vec;
template <>
struct Vec<__nv_bfloat16> {
    static constexpr int kN = 8;
    __device__ static void unpack(const uint4 w, float* v) {
        v[0] = bf16lo(w.x); v[1] = bf16hi(w.x);
        v[2] = bf16lo(w.y); v[3] = bf16hi(w.y);
        v[4] = bf16lo(w.z); v[5] = bf16hi(w.z);
        v[6] = bf16lo(w.w); v[7] = bf16hi(w.w);
    }
    __device__ static float load(const void* p) {
        return __uint_as_float(static_cast<uint32_t>(*static_cast<const uint16_t*>(p)) << 16);
    }
};
template <>
struct Vec<float> {
    static constexpr int kN = 4;
    __device__ static void unpack(const uint4 w, float* v) {
        v[0] = __uint_as_float(w.x); v[1] = __uint_as_float(w.y);
        v[2] = __uint_as_float(w.z); v[3] = __uint_as_float(w.w);
    }
    __device__ static float load(const void* p) { return *static_cast<const float*>(p); }
};

template <typename Elem>
__device__ void produce(const StatsArgs& a, StatsSmem& sm) {
    constexpr int kEsz = sizeof(Elem);
    long long n = 0;
    for (long long w = blockIdx.x; w < a.n_items; w += gridDim.x) {
        const int slot = static_cast<int>(w / a.nchunks);
        const int c = static_cast<int>(w - static_cast<long long>(slot) * a.nchunks);
        const int r = a.two_rows ? (slot >> 1) : slot;
        const int kind = a.two_rows ? (slot & 1) : 0;
        const int i = seq_of_position(a.seq_offsets, a.num_seqs, r);
        const SeqInfo s = seq_info(a.seq_offsets, a.temperature, i, a.total);
        if (!s.ok || r < s.start || r >= s.start + s.len) continue;
        if (kind == 1 && s.T == 0.0f) continue;  // greedy verification never reads q
        if (a.accept_len != nullptr && __ldg(a.accept_len + i) != s.len) continue;
        const long long row = kind ? r : (a.two_rows ? static_cast<long long>(r) + i : r);
        const char* base = kind ? a.rows1 + row * a.ld1_bytes : a.rows0 + row * a.ld0_bytes;
        const int e0 = c * a.chunk;
        const int n_el = min(a.chunk, a.vocab - e0);
        const uintptr_t start_b = reinterpret_cast<uintptr_t>(base) + static_cast<uintptr_t>(e0) * kEsz;
        const uintptr_t end_b = start_b + static_cast<uintptr_t>(n_el) * kEsz;
        const uintptr_t lo = start_b & ~static_cast<uintptr_t>(15);
        const uintptr_t hi = end_b & ~static_cast<uintptr_t>(15);
        ItemDesc d;
        d.slot = slot;
        d.chunk = c;
        d.end = 0;
        if (hi > lo) {
            d.tma_bytes = static_cast<int>(hi - lo);
            d.skip = static_cast<int>((start_b - lo) / kEsz);
            d.n_smem = static_cast<int>((hi - start_b) / kEsz);
        } else {
            d.tma_bytes = 0;
            d.skip = 0;
            d.n_smem = 0;
        }
        d.n_tail = n_el - d.n_smem;
        d.tail_src = reinterpret_cast<const char*>(start_b) + static_cast<size_t>(d.n_smem) * kEsz;
        d.c2 = s.T > 0.0f ? inv_temp_log2e(s.T) : 0.0f;
        d.gather = -1;
        if (a.tokens != nullptr) {  // both rows of a verified position score x_k
            const int g = __ldg(a.tokens + r) - e0;
            if (g >= 0 && g < n_el) d.gather = g;
        }
        const int stage = static_cast<int>(n % kStages);
        const uint32_t parity = (static_cast<uint32_t>(n / kStages) & 1u) ^ 1u;
        if (!mbar_wait(&sm.empty[stage], parity)) {
            atomicOr(a.err, kErrWaitTimeout);
            return;  // consumers time out on their own wait
        }
        sm.desc[stage] = d;
        if (d.tma_bytes > 0) {
            mbar_arrive_expect_tx(&sm.full[stage], static_cast<uint32_t>(d.tma_bytes));
            bulk_copy_g2s(sm.stage[stage], reinterpret_cast<const void*>(lo),
                          static_cast<uint32_t>(d.tma_bytes), &sm.full[stage]);
        } else {
            mbar_arrive(&sm.full[stage]);
        }
        ++n;
    }
    const int stage = static_cast<int>(n % kStages);
    const uint32_t parity = (static_cast<uint32_t>(n / kStages) & 1u) ^ 1u;
    if (!mbar_wait(&sm.empty[stage], parity)) {
        atomicOr(a.err, kErrWaitTimeout);
        return;
    }
    sm.desc[stage].end = 1;
    mbar_arrive(&sm.full[stage]);
}

template <typename Elem>
__device__ void consume(const StatsArgs& a, StatsSmem& sm, int tid, int warp, int lane) {
    constexpr int kEsz = sizeof(Elem);
    constexpr int kN = Vec<Elem>::kN;
    constexpr int kVals = kVecPerThread * kN;
    for (long long n = 0;; ++n) {
        const int stage = static_cast<int>(n % kStages);
        const uint32_t parity = static_cast<uint32_t>(n / kStages) & 1u;
        // A wait only gives up after a fault; the warp then skips the round
        // and the whole consumer group leaves together after the barrier.
        const bool ok = __all_sync(0xffffffffu, mbar_wait(&sm.full[stage], parity));
        if (!ok && lane == 0) {
            sm.abort = 1;
            atomicOr(a.err, kErrWaitTimeout);
        }
        ItemDesc d;
        d.end = 1;
        if (ok) d = sm.desc[stage];
        const int par = static_cast<int>(n & 1);

        if (ok && !d.end) {
            // Shared memory -> registers; the stage is then released.
            float v[kVals];
            const int nvec = d.tma_bytes >> 4;
            const uint4* sv = reinterpret_cast<const uint4*>(sm.stage[stage]);
#pragma unroll
            for (int k = 0; k < kVecPerThread; ++k) {
                const int vi = tid + k * kConsumerThreads;
                if (vi < nvec) {
                    Vec<Elem>::unpack(sv[vi], &v[k * kN]);
                    if (vi == 0) {
#pragma unroll
                        for (int j = 0; j < kN; ++j)
                            if (j < d.skip) v[j] = -INFINITY;
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < kN; ++j) v[k * kN + j] = -INFINITY;
                }
            }
            float tailv = -INFINITY;
            if (tid < d.n_tail) tailv = Vec<Elem>::load(d.tail_src + static_cast<size_t>(tid) * kEsz);
            float gathered = 0.0f;
            if (tid == 0 && d.gather >= 0) {
                gathered = d.gather < d.n_smem
                               ? Vec<Elem>::load(sm.stage[stage] + static_cast<size_t>(d.gather + d.skip) * kEsz)
                               : Vec<Elem>::load(d.tail_src + static_cast<size_t>(d.gather - d.n_smem) * kEsz);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.empty[stage]);

            // Thread, then warp partials.
            float m = tailv;
#pragma unroll
            for (int e = 0; e < kVals; ++e) m = fmaxf(m, v[e]);
            const float mw = warp_max(m);
            if (d.c2 > 0.0f) {
                float sum = 0.0f;
                if (mw != -INFINITY) {
#pragma unroll
                    for (int e = 0; e < kVals; ++e) sum += ex2_approx((v[e] - mw) * d.c2);
                    sum += ex2_approx((tailv - mw) * d.c2);
                }
                const float sw = warp_sum(sum);
                if (lane == 0) sm.red[par][warp] = make_float2(mw, sw);
            } else {
                int idx = INT_MAX;
                if (m == mw && mw != -INFINITY) {
                    // The first match in this thread's element order is its lowest id.
#pragma unroll
                    for (int k = kVecPerThread - 1; k >= 0; --k)
#pragma unroll
                        for (int j = kN - 1; j >= 0; --j)
                            if (v[k * kN + j] == mw) idx = (tid + k * kConsumerThreads) * kN + j - d.skip;
                    if (idx == INT_MAX && tailv == mw) idx = d.n_smem + tid;
                }
                const int iw = warp_min_int(idx);
                if (lane == 0) {
                    sm.red[par][warp] = make_float2(mw, 0.0f);
                    sm.redi[par][warp] = iw;
                }
            }
            if (tid == 0 && d.gather >= 0) a.zx[d.slot] = gathered;
        }
        named_barrier_sync(1, kConsumerThreads);
        if (sm.abort) {
            // Let copies still in flight land before the CTA's shared memory
            // is released (bounded waits on the stages that may hold one).
            if (tid == 0)
                for (int k = 0; k < kStages; ++k) {
                    const long long nn = n + k;
                    (void)mbar_wait(&sm.full[nn % kStages], static_cast<uint32_t>(nn / kStages) & 1u);
                }
            return;
        }
        if (d.end) return;  // every wait succeeded, so every thread read the same marker

        // Chunk partial from the eight warp partials.
        if (warp == 0) {
            const float2 pw = lane < kConsumerWarps ? sm.red[par][lane] : make_float2(-INFINITY, 0.0f);
            const float M = warp_max(pw.x);
            float2 out;
            if (d.c2 > 0.0f) {
                const float sc = (pw.x == -INFINITY) ? 0.0f : pw.y * exp2f((pw.x - M) * d.c2);
                out = make_float2(M, warp_sum(sc));
            } else {
                const int iw = lane < kConsumerWarps ? sm.redi[par][lane] : INT_MAX;
                const int I = warp_min_int(pw.x == M ? iw : INT_MAX);
                const int gid = I == INT_MAX ? INT_MAX : I + d.chunk * a.chunk;
                out = make_float2(M, __int_as_float(gid));
            }
            if (lane == 0) a.part[static_cast<size_t>(d.slot) * a.nchunks + d.chunk] = out;
        }
    }
}

template <typename Elem>
__global__ void __launch_bounds__(kStatsThreads, kStatsCtasPerSm) stats_kernel(const StatsArgs a) {
    extern __shared__ unsigned char smem_raw[];
    StatsSmem& sm = *reinterpret_cast<StatsSmem*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~static_cast<uintptr_t>(127));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    pdl_wait();
    pdl_launch_dependents();
    for (int z = blockIdx.x * blockDim.x + tid; z < a.zero_count; z += gridDim.x * blockDim.x)
        a.zero_ptr[z] = 0;
    if (tid == 0) {
        sm.abort = 0;
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], kConsumerWarps);
        }
        fence_mbarrier_init();
    }
    __syncthreads();
    if (warp == kConsumerWarps) {
        if (lane == 0) produce<Elem>(a, sm);
        return;
    }
    consume<Elem>(a, sm, tid, warp, lane);
}

template <typename Elem>
cudaError_t launch_stats_t(const StatsArgs& a, int grid, cudaStream_t stream) {
    const size_t smem = sizeof(StatsSmem) + 128;
    cudaError_t err = cudaFuncSetAttribute(stats_kernel<Elem>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    stats_kernel<Elem><<<grid, kStatsThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_stats(const StatsArgs& a, int elem_bytes, int grid, cudaStream_t stream) {
    return elem_bytes == 2 ? launch_stats_t<__nv_bfloat16>(a, grid, stream)
                           : launch_stats_t<float>(a, grid, stream);
}

}  // namespace isd
