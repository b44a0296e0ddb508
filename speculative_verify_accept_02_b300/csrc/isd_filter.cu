// Verify and propose under the sampling filters of the pages' evaluation
// setting ("Introspective Diffusion Language Models | Summary", experiments
// §4.1: top-k 50, top-p 0.95 at temperature 1), applied to p and q before
// the ratio, the residual and every draw (§3.2's rules on the filtered
// distributions).
//
// A filtered distribution is fixed by the row's k best logits alone: the
// kept probabilities are renormalised over the kept ids, so the row's full
// softmax normaliser cancels.  Each call therefore runs two kernels:
//   topk_rows_kernel  one CTA per row streams the row once with 16-byte
//                     loads, four in flight per lane; every warp keeps a
//                     sorted list of its 64 best
//                     (logit, id) pairs in registers (two per lane) and
//                     inserts the rare candidate that beats its k-th entry;
//                     warp 0 merges the eight lists and writes the row's k
//                     best, ordered by logit (lower id first among equals);
//   filtered_*_kernel one warp per sequence reads those lists, applies the
//                     top-p cut, and takes every decision and draw: ratios,
//                     the accept prefix, the residual over at most k ids,
//                     inverse-CDF draws in vocabulary order, proposals.
// No kernel waits on another CTA; the second launch follows the first on
// the caller's stream.
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>

#include "../../include/isd_filter.h"
#include "isd_device.cuh"

namespace isd {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kListMax = ISD_FILTER_MAX_TOP_K;  // two entries per lane
static_assert(kListMax == 64, "a warp list holds two entries per lane");
constexpr int kTopkThreads = 256;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kTopkCtasPerSm = 4;
constexpr int kInFlight = 4;  // 16-byte loads in flight per lane of topk_rows_kernel
constexpr int kSeqThreads = 256;
constexpr int kSeqWarps = kSeqThreads / 32;
constexpr double kLog2eD = 1.4426950408889634;  // log2(e)

// Rank order of (logit, id) pairs: larger logit first, lower id among equals.
__device__ __forceinline__ bool beats(float av, int ai, float bv, int bi) {
    return av > bv || (av == bv && ai < bi);
}

// A warp's sorted list of its 64 best (logit, id) pairs: lane j holds
// entries 2j (v0, i0) and 2j+1 (v1, i1).  Empty entries are (-inf, INT_MAX),
// which every real element beats or ties below.
struct WarpList {
    float v0, v1;
    int i0, i1;

    __device__ void init() {
        v0 = v1 = -INFINITY;
        i0 = i1 = INT_MAX;
    }

    // Entry j (the same j in every lane), broadcast.
    __device__ void get(int j, float& v, int& id) const {
        v = __shfl_sync(kFull, (j & 1) ? v1 : v0, j >> 1);
        id = __shfl_sync(kFull, (j & 1) ? i1 : i0, j >> 1);
    }

    // Inserts (cv, ci) at its rank; entries past index 63 fall off.  Called
    // by the whole warp with the same candidate.
    __device__ void insert(float cv, int ci, int lane) {
        const int pos = __popc(__ballot_sync(kFull, beats(v0, i0, cv, ci))) +
                        __popc(__ballot_sync(kFull, beats(v1, i1, cv, ci)));
        const float pv = __shfl_up_sync(kFull, v1, 1);  // entry 2j - 1
        const int pi = __shfl_up_sync(kFull, i1, 1);
        const int e0 = 2 * lane, e1 = 2 * lane + 1;
        float nv1 = v1, nv0 = v0;
        int ni1 = i1, ni0 = i0;
        if (e1 > pos) {
            nv1 = v0;
            ni1 = i0;
        } else if (e1 == pos) {
            nv1 = cv;
            ni1 = ci;
        }
        if (e0 > pos) {
            nv0 = pv;
            ni0 = pi;
        } else if (e0 == pos) {
            nv0 = cv;
            ni0 = ci;
        }
        v0 = nv0;
        i0 = ni0;
        v1 = nv1;
        i1 = ni1;
    }
};

// Offers each lane's candidate (if `has`) to the list; (tv, ti) is the
// list's entry k - 1, the bar a candidate must beat.
__device__ __forceinline__ void offer(WarpList& wl, float cv, int ci, bool has, int k, float& tv, int& ti,
                                      int lane) {
    unsigned m = __ballot_sync(kFull, has && beats(cv, ci, tv, ti));
    while (m) {
        const int src = __ffs(m) - 1;
        m &= m - 1;
        const float v = __shfl_sync(kFull, cv, src);
        const int id = __shfl_sync(kFull, ci, src);
        if (beats(v, id, tv, ti)) {
            wl.insert(v, id, lane);
            wl.get(k - 1, tv, ti);
        }
    }
}

struct TopkArgs {
    const char* base[3];   // row buffers (p, q) or (qnew)
    int64_t ld_bytes[3];
    int nrows[3];
    int nbuf;
    int vocab;
    int k;                 // entries kept per row, 1..64
    float* out_v;          // [rows][k]
    int* out_i;            // [rows][k]
};

template <int E>
__global__ void __launch_bounds__(kTopkThreads) topk_rows_kernel(TopkArgs a) {
    constexpr int VEC = 16 / E;
    __shared__ float s_v[kTopkWarps][kListMax];
    __shared__ int s_i[kTopkWarps][kListMax];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // rows of buffer 0, then 1, then 2 (selects, not indexing: the argument
    // arrays stay in the constant bank)
    const long long n0 = a.nrows[0], n1 = a.nbuf > 1 ? a.nrows[1] : 0, n2 = a.nbuf > 2 ? a.nrows[2] : 0;
    const long long rows = n0 + n1 + n2;
    const int V = a.vocab, k = a.k;
    for (long long r = blockIdx.x; r < rows; r += gridDim.x) {
        const char* row;
        if (r < n0)
            row = a.base[0] + r * a.ld_bytes[0];
        else if (r < n0 + n1)
            row = a.base[1] + (r - n0) * a.ld_bytes[1];
        else
            row = a.base[2] + (r - n0 - n1) * a.ld_bytes[2];
        const uintptr_t mis = reinterpret_cast<uintptr_t>(row) & 15u;
        const int head = min(V, mis ? static_cast<int>((16u - mis) / E) : 0);
        const int nvec = (V - head) / VEC;
        const int tail0 = head + nvec * VEC;
        WarpList wl;
        wl.init();
        float tv = -INFINITY;
        int ti = INT_MAX;
        const uint4* body = reinterpret_cast<const uint4*>(row + static_cast<size_t>(head) * E);
        // kInFlight vectors per lane are loaded ahead of the one being
        // offered: each slot is refilled with the vector kInFlight steps on
        // as soon as it is taken.
        uint4 ahead[kInFlight];
#pragma unroll
        for (int d = 0; d < kInFlight; ++d) {
            const int g = warp * 32 + d * kTopkThreads + lane;
            ahead[d] = g < nvec ? __ldg(body + g) : make_uint4(0u, 0u, 0u, 0u);
        }
        for (int g0 = warp * 32; g0 < nvec; g0 += kInFlight * kTopkThreads) {
#pragma unroll
            for (int d = 0; d < kInFlight; ++d) {
                const int gs = g0 + d * kTopkThreads;  // the warp's first vector of this step
                if (gs >= nvec) break;                // the same for every lane
                const int g = gs + lane;
                const bool has = g < nvec;
                const uint4 w = ahead[d];
                const int gn = g + kInFlight * kTopkThreads;
                ahead[d] = gn < nvec ? __ldg(body + gn) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                for (int j = 0; j < VEC; ++j)
                    offer(wl, vec_elem<E>(w, j), head + g * VEC + j, has, k, tv, ti, lane);
            }
        }
        if (warp == 0) {  // the unaligned head and the tail: fewer than 2 * VEC ids
            const int e = lane < head ? lane : tail0 + (lane - head);
            const bool has = lane < head || (lane - head < V - tail0);
            float v = -INFINITY;
            if (has) {
                const char* p = row + static_cast<size_t>(e) * E;
                if constexpr (E == 2)
                    v = __uint_as_float(static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short*>(p))) << 16);
                else
                    v = __ldg(reinterpret_cast<const float*>(p));
            }
            offer(wl, v, e, has, k, tv, ti, lane);
        }
        // Merge: every warp's first k entries into warp 0's list.
        if (2 * lane < k) {
            s_v[warp][2 * lane] = wl.v0;
            s_i[warp][2 * lane] = wl.i0;
        }
        if (2 * lane + 1 < k) {
            s_v[warp][2 * lane + 1] = wl.v1;
            s_i[warp][2 * lane + 1] = wl.i1;
        }
        __syncthreads();
        if (warp == 0) {
            for (int w = 1; w < kTopkWarps; ++w)
                for (int j = 0; j < k; ++j) {
                    const float cv = s_v[w][j];
                    const int ci = s_i[w][j];
                    if (!beats(cv, ci, tv, ti)) break;  // each list is sorted: the rest cannot
                    wl.insert(cv, ci, lane);
                    wl.get(k - 1, tv, ti);
                }
            float* ov = a.out_v + r * k;
            int* oi = a.out_i + r * k;
            if (2 * lane < k) {
                ov[2 * lane] = wl.v0;
                oi[2 * lane] = wl.i0;
            }
            if (2 * lane + 1 < k) {
                ov[2 * lane + 1] = wl.v1;
                oi[2 * lane + 1] = wl.i1;
            }
        }
        __syncthreads();  // s_v, s_i are rewritten for the next row
    }
}

// ---------------------------------------------------------------------------
// Filtered distributions from the lists (one warp)
// ---------------------------------------------------------------------------

// The arithmetic on the lists runs in double precision: it is at most 64
// values per row, so it costs little even at fp64 rates, and it keeps the
// top-p cut, the ratios and the draws within rounding of their definitions.
__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}

__device__ __forceinline__ double warp_inclusive_scan_d(double v, int lane) {
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const double y = __shfl_up_sync(kFull, v, d);
        if (lane >= d) v += y;
    }
    return v;
}

// The filtered probabilities of one list row: lane j holds entries 2j and
// 2j+1 (ids and p~, 0 past the top-p cut or the list).
struct FRow {
    int id0, id1;
    double p0, p1;
};

// c2 = log2(e) / T.
__device__ FRow filtered_row(const float* lv, const int* li, long long r, int k, double c2, double top_p,
                             int lane) {
    FRow f;
    const int j0 = 2 * lane, j1 = j0 + 1;
    const float* v = lv + r * k;
    const int* id = li + r * k;
    const float z0 = j0 < k ? __ldg(v + j0) : -INFINITY;
    const float z1 = j1 < k ? __ldg(v + j1) : -INFINITY;
    f.id0 = j0 < k ? __ldg(id + j0) : INT_MAX;
    f.id1 = j1 < k ? __ldg(id + j1) : INT_MAX;
    const double zmax = __ldg(v);  // the list's first entry is its largest logit
    // weights proportional to softmax(z / T) over the list; -inf entries weigh 0
    const double w0 = z0 == -INFINITY ? 0.0 : exp2((static_cast<double>(z0) - zmax) * c2);
    const double w1 = z1 == -INFINITY ? 0.0 : exp2((static_cast<double>(z1) - zmax) * c2);
    const double pair = w0 + w1;
    const double incl = warp_inclusive_scan_d(pair, lane);
    const double sk = __shfl_sync(kFull, incl, 31);
    int n = k;
    if (top_p < 1.0) {  // shortest prefix whose share of the top-k mass reaches top_p
        const double c0 = incl - pair + w0;
        int first = INT_MAX;
        if (j1 < k && incl / sk >= top_p) first = j1;
        if (j0 < k && c0 / sk >= top_p) first = j0;
        first = warp_min_int(first);
        n = first == INT_MAX ? k : first + 1;
    }
    const double k0 = j0 < n ? w0 : 0.0, k1 = j1 < n ? w1 : 0.0;
    const double total = warp_sum_d(k0 + k1);
    f.p0 = k0 / total;
    f.p1 = k1 / total;
    return f;
}

// p~(x) of one filtered row (0 if x is not kept).
__device__ __forceinline__ double prob_of(const FRow& f, int x) {
    double v = 0.0;
    if (f.id0 == x) v = f.p0;
    if (f.id1 == x) v = f.p1;
    return warp_sum_d(v);  // ids are distinct: at most one lane contributes
}

// Inverse-CDF draw in vocabulary order over a warp's 64 (id, weight)
// entries: with S the sum of the weights and t = u*S, the smallest id whose
// running sum exceeds t; if rounding leaves none, the largest id of positive
// weight.  `sid`, `sw`: this warp's 64-entry scratch in shared memory.
__device__ int warp_icdf(int id0, double w0, int id1, double w1, float u, int* sid, double* sw, int lane) {
    // rank of each entry in (id, list index) order
    int r0 = 0, r1 = 0;
    const int j0 = 2 * lane, j1 = j0 + 1;
    for (int t = 0; t < 32; ++t) {
        const int a0 = __shfl_sync(kFull, id0, t), a1 = __shfl_sync(kFull, id1, t);
        const int t0 = 2 * t, t1 = t0 + 1;
        r0 += (a0 < id0 || (a0 == id0 && t0 < j0)) + (a1 < id0 || (a1 == id0 && t1 < j0));
        r1 += (a0 < id1 || (a0 == id1 && t0 < j1)) + (a1 < id1 || (a1 == id1 && t1 < j1));
    }
    __syncwarp();
    sid[r0] = id0;
    sw[r0] = w0;
    sid[r1] = id1;
    sw[r1] = w1;
    __syncwarp();
    const int s0 = sid[j0], s1 = sid[j1];
    const double x0 = sw[j0], x1 = sw[j1];
    __syncwarp();
    const double pair = x0 + x1;
    const double incl = warp_inclusive_scan_d(pair, lane);
    const double S = __shfl_sync(kFull, incl, 31);
    const double t = static_cast<double>(u) * S;
    const double c0 = incl - pair + x0;
    int first = INT_MAX;
    if (incl > t) first = j1;
    if (c0 > t) first = j0;
    first = warp_min_int(first);
    if (first == INT_MAX) {
        int last = -1;
        if (x0 > 0.0) last = j0;
        if (x1 > 0.0) last = j1;
        first = warp_max_int(last);
        if (first < 0) return -1;
    }
    const int tok = (first & 1) ? s1 : s0;
    return __shfl_sync(kFull, tok, first >> 1);
}

// ---------------------------------------------------------------------------
// Verify: one warp per sequence
// ---------------------------------------------------------------------------

struct FiltVerifyArgs {
    const float* lv;   // lists: rows [0, total + C) are p rows, then total q rows
    const int* li;
    int k;
    float top_p;
    int vocab;
    const int32_t* tokens;
    const int32_t* offs;
    int num_seqs;
    int total;
    const float* temp;
    uint64_t seed, offset;
    int32_t* accept_len;
    int32_t* out_tokens;
    float* ratio;
    float* alpha;
};

__global__ void __launch_bounds__(kSeqThreads) filtered_verify_kernel(FiltVerifyArgs a) {
    __shared__ int s_id[kSeqWarps][kListMax];
    __shared__ double s_w[kSeqWarps][kListMax];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const long long qbase = static_cast<long long>(a.total) + a.num_seqs;
    for (int i = blockIdx.x * kSeqWarps + warp; i < a.num_seqs; i += gridDim.x * kSeqWarps) {
        const SeqInfo s = seq_info(a.offs, a.temp, i, a.total);
        const int L = s.len;
        const bool mine = s.ok && lane < L;
        const int x = mine ? __ldg(a.tokens + s.start + lane) : 0;
        const bool bad_tok = __any_sync(kFull, mine && (x < 0 || x >= a.vocab));
        if (!s.ok || bad_tok) {
            if (s.in_range) {
                for (int m = lane; m <= L; m += 32) a.out_tokens[s.start + i + m] = -1;
                for (int m = lane; m < L; m += 32) a.ratio[s.start + m] = NAN;
            }
            if (lane == 0) {
                a.accept_len[i] = -1;
                a.alpha[i] = NAN;
            }
            continue;
        }
        const long long prow0 = static_cast<long long>(s.start) + i;  // p row of position 1
        double my_ratio = 0.0;
        int acc_len, token;
        if (s.T == 0.0f) {  // greedy: the lists' first ids are the (lowest-id) argmaxes
            if (mine) my_ratio = x == __ldg(a.li + (prow0 + lane) * a.k) ? 1.0 : 0.0;
            const unsigned fail = __ballot_sync(kFull, mine && my_ratio == 0.0);
            acc_len = fail ? __ffs(fail) - 1 : L;
            token = __ldg(a.li + (prow0 + acc_len) * a.k);
        } else {
            const double c2 = kLog2eD / static_cast<double>(s.T);
            const double top_p = a.top_p;
            for (int kk = 0; kk < L; ++kk) {
                const int xk = __shfl_sync(kFull, x, kk);
                const FRow P = filtered_row(a.lv, a.li, prow0 + kk, a.k, c2, top_p, lane);
                const FRow Q = filtered_row(a.lv, a.li, qbase + s.start + kk, a.k, c2, top_p, lane);
                const double px = prob_of(P, xk), qx = prob_of(Q, xk);
                const double rk = qx == 0.0 ? 1.0 : fmin(1.0, px / qx);
                if (lane == kk) my_ratio = rk;
            }
            bool accepted = false;
            if (mine)
                accepted = static_cast<double>(decision_uniform(a.seed, a.offset, i, lane + 1, kTagAccept)) < my_ratio;
            const unsigned fail = __ballot_sync(kFull, mine && !accepted);
            acc_len = fail ? __ffs(fail) - 1 : L;
            const FRow P = filtered_row(a.lv, a.li, prow0 + acc_len, a.k, c2, top_p, lane);
            double w0 = P.p0, w1 = P.p1;
            float u;
            if (acc_len < L) {  // residual normalize(max(0, p~ - q~)), over p~'s kept ids
                const FRow Q = filtered_row(a.lv, a.li, qbase + s.start + acc_len, a.k, c2, top_p, lane);
                double q0 = 0.0, q1 = 0.0;
                for (int t = 0; t < 32; ++t) {
                    const int b0 = __shfl_sync(kFull, Q.id0, t), b1 = __shfl_sync(kFull, Q.id1, t);
                    const double y0 = __shfl_sync(kFull, Q.p0, t), y1 = __shfl_sync(kFull, Q.p1, t);
                    if (b0 == P.id0) q0 = y0;
                    if (b1 == P.id0) q0 = y1;
                    if (b0 == P.id1) q1 = y0;
                    if (b1 == P.id1) q1 = y1;
                }
                const double r0 = fmax(0.0, P.p0 - q0), r1 = fmax(0.0, P.p1 - q1);
                if (warp_sum_d(r0 + r1) > 0.0) {
                    w0 = r0;
                    w1 = r1;
                }
                u = decision_uniform(a.seed, a.offset, i, acc_len + 1, kTagCorrect);
            } else {  // bonus token from the final anchor p~_{L+1}
                u = decision_uniform(a.seed, a.offset, i, L + 1, kTagBonus);
            }
            token = warp_icdf(P.id0, w0, P.id1, w1, u, s_id[warp], s_w[warp], lane);
        }
        if (mine) a.ratio[s.start + lane] = static_cast<float>(my_ratio);
        const double sum = warp_sum_d(mine ? my_ratio : 0.0);
        // slot m < 32 belongs to lane m, whose x is x_{m+1}; slot 32 (L = 32) is never a proposal
        for (int m = lane; m <= L; m += 32)
            a.out_tokens[s.start + i + m] = m < acc_len ? x : (m == acc_len ? token : -1);
        if (lane == 0) {
            a.accept_len[i] = acc_len;
            a.alpha[i] = static_cast<float>(sum / L);
        }
    }
}

// ---------------------------------------------------------------------------
// Propose: one warp per sequence
// ---------------------------------------------------------------------------

struct FiltProposeArgs {
    const float* lv;   // lists of the qnew rows
    const int* li;
    int k;
    float top_p;
    const int32_t* offs;
    int num_seqs;
    int total;
    const float* temp;
    const int32_t* accept_len;  // optional
    uint64_t seed, offset;
    int32_t* proposals;
    uint8_t* valid;
};

__global__ void __launch_bounds__(kSeqThreads) filtered_propose_kernel(FiltProposeArgs a) {
    __shared__ int s_id[kSeqWarps][kListMax];
    __shared__ double s_w[kSeqWarps][kListMax];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int i = blockIdx.x * kSeqWarps + warp; i < a.num_seqs; i += gridDim.x * kSeqWarps) {
        const SeqInfo s = seq_info(a.offs, a.temp, i, a.total);
        bool draw = s.ok;
        if (draw && a.accept_len != nullptr) draw = __ldg(a.accept_len + i) == s.len;
        if (lane == 0) a.valid[i] = draw ? 1 : 0;
        if (!draw) {
            if (s.in_range)
                for (int m = lane; m < s.len; m += 32) a.proposals[s.start + m] = -1;
            continue;
        }
        const double c2 = s.T > 0.0f ? kLog2eD / static_cast<double>(s.T) : 0.0;
        for (int m = 0; m < s.len; ++m) {
            const long long r = static_cast<long long>(s.start) + m;
            int tok;
            if (s.T == 0.0f) {
                tok = __ldg(a.li + r * a.k);
            } else {
                const FRow F = filtered_row(a.lv, a.li, r, a.k, c2, static_cast<double>(a.top_p), lane);
                const float u = decision_uniform(a.seed, a.offset, i, m + 1, kTagPropose);
                tok = warp_icdf(F.id0, F.p0, F.id1, F.p1, u, s_id[warp], s_w[warp], lane);
            }
            if (lane == 0) a.proposals[r] = tok;
        }
    }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

constexpr size_t kAlign = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Lists of `rows` rows: values, then ids.
size_t list_bytes(long long rows, int k) {
    return align_up(static_cast<size_t>(rows) * k * sizeof(float)) + align_up(static_cast<size_t>(rows) * k * sizeof(int));
}

bool filter_ok(int top_k, float top_p) {
    return top_k >= 1 && top_k <= ISD_FILTER_MAX_TOP_K && std::isfinite(top_p) && top_p > 0.0f && top_p <= 1.0f;
}

isd_status grid_for(long long items, int per_sm, int* grid) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return ISD_ERR_CUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return ISD_ERR_CUDA;
    long long g = static_cast<long long>(sms) * per_sm;
    if (items < g) g = items;
    *grid = static_cast<int>(g < 1 ? 1 : g);
    return ISD_OK;
}

isd_status launch_topk(const TopkArgs& t, int esz, cudaStream_t stream) {
    long long rows = 0;
    for (int b = 0; b < t.nbuf; ++b) rows += t.nrows[b];
    if (rows == 0) return ISD_OK;  // nothing to select; the second kernel reads no list
    int grid = 1;
    const isd_status gs = grid_for(rows, kTopkCtasPerSm, &grid);
    if (gs != ISD_OK) return gs;
    if (esz == 2)
        topk_rows_kernel<2><<<grid, kTopkThreads, 0, stream>>>(t);
    else
        topk_rows_kernel<4><<<grid, kTopkThreads, 0, stream>>>(t);
    return cudaGetLastError() == cudaSuccess ? ISD_OK : ISD_ERR_CUDA;
}

}  // namespace
}  // namespace isd

extern "C" {

size_t isd_verify_filtered_workspace_bytes(int num_seqs, int total_positions, int top_k) {
    if (num_seqs < 0 || total_positions < 0 || top_k < 1 || top_k > ISD_FILTER_MAX_TOP_K) return 0;
    return isd::list_bytes(2LL * total_positions + num_seqs, top_k);
}

size_t isd_propose_filtered_workspace_bytes(int num_seqs, int total_positions, int top_k) {
    if (num_seqs < 0 || total_positions < 0 || top_k < 1 || top_k > ISD_FILTER_MAX_TOP_K) return 0;
    return isd::list_bytes(total_positions, top_k);
}

isd_status isd_verify_filtered(const void* p_logits, int64_t ld_p, const void* q_logits, int64_t ld_q,
                               isd_dtype dtype, int vocab, const int32_t* tokens, const int32_t* seq_offsets,
                               int num_seqs, int total_positions, const float* temperature, uint64_t seed,
                               uint64_t offset, int top_k, float top_p, int32_t* accept_len, int32_t* out_tokens,
                               float* ratio, float* alpha, void* workspace, size_t workspace_bytes, void* stream) {
    if (num_seqs < 0 || total_positions < 0 || vocab < 1 || (dtype != ISD_DTYPE_BF16 && dtype != ISD_DTYPE_F32))
        return ISD_ERR_INVALID_ARG;
    if (!isd::filter_ok(top_k, top_p)) return ISD_ERR_INVALID_ARG;
    if (num_seqs == 0) return ISD_OK;
    if (!p_logits || !q_logits || !tokens || !seq_offsets || !temperature || !accept_len || !out_tokens ||
        !ratio || !alpha || !workspace)
        return ISD_ERR_INVALID_ARG;
    if (ld_p < vocab || ld_q < vocab) return ISD_ERR_INVALID_ARG;
    if (!isd::aligned16(p_logits) || !isd::aligned16(q_logits)) return ISD_ERR_UNSUPPORTED;
    const long long rows = 2LL * total_positions + num_seqs;
    if (workspace_bytes < isd::list_bytes(rows, top_k) ||
        (reinterpret_cast<uintptr_t>(workspace) % isd::kAlign) != 0)
        return ISD_ERR_WORKSPACE;
    const int esz = dtype == ISD_DTYPE_BF16 ? 2 : 4;
    const int k = top_k < vocab ? top_k : vocab;
    char* ws = static_cast<char*>(workspace);
    float* lv = reinterpret_cast<float*>(ws);
    int* li = reinterpret_cast<int*>(ws + isd::align_up(static_cast<size_t>(rows) * k * sizeof(float)));
    isd::TopkArgs t{};
    t.base[0] = static_cast<const char*>(p_logits);
    t.ld_bytes[0] = ld_p * esz;
    t.nrows[0] = total_positions + num_seqs;
    t.base[1] = static_cast<const char*>(q_logits);
    t.ld_bytes[1] = ld_q * esz;
    t.nrows[1] = total_positions;
    t.nbuf = 2;
    t.vocab = vocab;
    t.k = k;
    t.out_v = lv;
    t.out_i = li;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    const isd_status ts = isd::launch_topk(t, esz, st);
    if (ts != ISD_OK) return ts;
    isd::FiltVerifyArgs f{};
    f.lv = lv;
    f.li = li;
    f.k = k;
    f.top_p = top_p;
    f.vocab = vocab;
    f.tokens = tokens;
    f.offs = seq_offsets;
    f.num_seqs = num_seqs;
    f.total = total_positions;
    f.temp = temperature;
    f.seed = seed;
    f.offset = offset;
    f.accept_len = accept_len;
    f.out_tokens = out_tokens;
    f.ratio = ratio;
    f.alpha = alpha;
    const int grid = (num_seqs + isd::kSeqWarps - 1) / isd::kSeqWarps;
    isd::filtered_verify_kernel<<<grid, isd::kSeqThreads, 0, st>>>(f);
    return cudaGetLastError() == cudaSuccess ? ISD_OK : ISD_ERR_CUDA;
}

isd_status isd_propose_filtered(const void* qnew_logits, int64_t ld, isd_dtype dtype, int vocab,
                                const int32_t* seq_offsets, int num_seqs, int total_positions,
                                const float* temperature, uint64_t seed, uint64_t offset, int top_k, float top_p,
                                const int32_t* accept_len_or_null, int32_t* proposals, uint8_t* valid,
                                void* workspace, size_t workspace_bytes, void* stream) {
    if (num_seqs < 0 || total_positions < 0 || vocab < 1 || (dtype != ISD_DTYPE_BF16 && dtype != ISD_DTYPE_F32))
        return ISD_ERR_INVALID_ARG;
    if (!isd::filter_ok(top_k, top_p)) return ISD_ERR_INVALID_ARG;
    if (num_seqs == 0) return ISD_OK;
    if (!qnew_logits || !seq_offsets || !temperature || !proposals || !valid || !workspace)
        return ISD_ERR_INVALID_ARG;
    if (ld < vocab) return ISD_ERR_INVALID_ARG;
    if (!isd::aligned16(qnew_logits)) return ISD_ERR_UNSUPPORTED;
    if (workspace_bytes < isd::list_bytes(total_positions, top_k) ||
        (reinterpret_cast<uintptr_t>(workspace) % isd::kAlign) != 0)
        return ISD_ERR_WORKSPACE;
    const int esz = dtype == ISD_DTYPE_BF16 ? 2 : 4;
    const int k = top_k < vocab ? top_k : vocab;
    char* ws = static_cast<char*>(workspace);
    float* lv = reinterpret_cast<float*>(ws);
    int* li = reinterpret_cast<int*>(ws + isd::align_up(static_cast<size_t>(total_positions) * k * sizeof(float)));
    isd::TopkArgs t{};
    t.base[0] = static_cast<const char*>(qnew_logits);
    t.ld_bytes[0] = ld * esz;
    t.nrows[0] = total_positions;
    t.nbuf = 1;
    t.vocab = vocab;
    t.k = k;
    t.out_v = lv;
    t.out_i = li;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    const isd_status ts = isd::launch_topk(t, esz, st);
    if (ts != ISD_OK) return ts;
    isd::FiltProposeArgs f{};
    f.lv = lv;
    f.li = li;
    f.k = k;
    f.top_p = top_p;
    f.offs = seq_offsets;
    f.num_seqs = num_seqs;
    f.total = total_positions;
    f.temp = temperature;
    f.accept_len = accept_len_or_null;
    f.seed = seed;
    f.offset = offset;
    f.proposals = proposals;
    f.valid = valid;
    const int grid = (num_seqs + isd::kSeqWarps - 1) / isd::kSeqWarps;
    isd::filtered_propose_kernel<<<grid, isd::kSeqThreads, 0, st>>>(f);
    return cudaGetLastError() == cudaSuccess ? ISD_OK : ISD_ERR_CUDA;
}

}  // extern "C"
