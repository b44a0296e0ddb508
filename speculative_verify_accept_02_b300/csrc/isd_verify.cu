// The verify step of Introspective Strided Decoding as one persistent kernel
// ("Introspective Diffusion Language Models | Summary", §2 acceptance rate,
// §3.2 strict acceptance, residual correction and bonus token, §3.3 online
// softmax over the vocabulary and a common acceptance path free of
// correction work), optionally with the next stride's proposal draws of the
// fused step (§3.2: one forward verifies and proposes).
//
// Work is handed out dynamically, in sequence order, by a global counter:
//   main item   one segment (up to eight 16 KB sub-chunks) of one p_k or q_k
//               row; greedy sequences stream their final anchor p_{L+1} in
//               place of their (unread) last q row.
//   decision    once a sequence's last item is done: ratio_k =
//               min(1, p_k(x_k) / q_k(x_k)), alpha, the accept prefix
//               (Philox uniforms, one warp ballot; relaxed acceptance tests
//               min(1, (1 + tau) p/q)) and the emitted prefix.  A greedy
//               correction or bonus is complete here (argmaxes of the
//               partials).
//   tail task   otherwise the decision publishes tails on a device queue: the
//               residual max(0, p_j - q_j) of the one rejected row pair, or
//               the final anchor row p_{L+1}; in the fused call also one per
//               qnew row of a sequence that accepted its whole stride.
//               Producers take queued tail tasks before new main items.
//   selection   once a tail's last task is done: the draw by inverse CDF, a
//               slice of about 500 ids from the tail partials, then an
//               in-order scan of that one slice (an argmax merge at T = 0).
//
// Warp roles of a CTA:
//   scheduler   (one thread) takes work: the next main item from the global
//               counter into a 2-entry work ring, a published tail task into
//               a priority slot; it absorbs every global memory round trip;
//   issuer      (one thread) streams the scheduled sub-chunks into a 4-stage
//               shared-memory ring with 1-D bulk copies under L2 eviction
//               policies, serving the priority slot between any two
//               sub-chunks; it never waits on global memory;
//   consumers   (8 warps) fold each stage into per-thread online softmax
//               partials (packed bf16 maxima, packed fp32 FMAs, one ex2 per
//               logit) or an exact argmax; at the end of an item every warp
//               hands its warp partial to the bookkeeper through a record
//               ring and moves on: consumers never wait on each other or on
//               global memory;
//   bookkeeper  (one warp) merges the records in batches, stores partials and
//               counts finished items per sequence with device-scope atomics;
//   finishers   (two warps) run the decisions and selections it triggers.
// The grid exits once every sequence is final; its last CTA re-zeroes the
// control block for the next call.  Every wait is bounded by the global timer.
#include <climits>
#include <type_traits>

#include "isd_device.cuh"
#include "isd_internal.h"

namespace isd {
namespace {

constexpr int kCW = 8;                    // consumer warps
constexpr int kCT = kCW * 32;             // consumer threads
constexpr int kIssuerWarp = kCW;
constexpr int kBookWarp = kCW + 1;
constexpr int kSchedWarp = kCW + 2;
constexpr int kFinWarp = kCW + 3;         // first of kFinishers finisher warps
constexpr int kFinishers = 2;
constexpr int kThreadsV = kCT + 32 * (3 + kFinishers);  // + issuer, bookkeeper, scheduler, finishers
constexpr int kStagesV = 4;
constexpr int kJobs = 16;                 // job ring between bookkeeper and finisher
constexpr int kWork = 2;                  // work ring between scheduler and issuer
constexpr int kRecs = 8;                  // record ring between consumers and bookkeeper
constexpr int kVecPT = kStageBytes / 16 / kCT;  // 16-byte vectors per consumer thread per stage
constexpr int kHalf = kStageBytes / 2;          // tail stages: [p piece | q piece]
constexpr int kSmemSeqs = 512;                  // batches up to this size keep offsets in shared memory
constexpr int kSmemToks = 2048;                 // batches up to this many positions keep their tokens there
constexpr int kSliceMax = 512;                  // ids in one tail slice (tail sub-chunk / 8 warps)
static_assert(kHalf / 2 <= kSliceMax * kCW, "a tail sub-chunk of bf16 ids splits into slices of at most kSliceMax");
static_assert(kVecPT * 16 * kCT == kStageBytes, "stage split");
static_assert(kHalf / kCW <= kSliceMax * 2, "a slice fits its staging buffer");
static_assert(kHalf / kCW <= 64 * 16, "a tail slice is at most two 16-byte vectors per lane");

enum : int { kEnd = 0, kMain = 1 };  // descriptor / record kinds besides the TailMode values
enum : int { kFirst = 1, kLast = 2 };

struct Desc {
    int kind;
    int flags;
    int seq;
    int slot;      // main: row slot (2 r + {0: p, 1: q}); tail: tail sub-chunk
    int seg;
    int expect;    // main: items of the sequence
    int e0;        // first element of the sub-chunk in its row
    int n;         // elements of the sub-chunk
    int nvec;      // main: 16-byte vectors in the stage
    int nsm0, skip0, nsm1, skip1;
    const char* tail0;  // global address of the first element not in shared memory
    const char* tail1;
    float c2, nz0, nz1;
};

// flags of a main record: which partial the warps hand in.
enum : int { kRecSoft = 0, kRecArg = 1 };

struct Rec {
    int kind, flags, seq, slot, seg, expect;
    float2 wp[kCW];  // one partial per consumer warp
};

// One unit of scheduled streaming: sub-chunks [c0, c1) of one row (main item)
// or of a tail row (pair).
struct Work {
    int kind;
    int seq, slot, seg, expect, c0, c1;
    int keep;  // load under the L2 evict_last policy (rows likely re-read by a tail)
    float c2, nz0, nz1;
    const char* row0;
    const char* row1;
};

// A finisher job: decide or select one sequence, or stop.
enum : int { kJobEnd = 0, kJobDecide = 1, kJobSelect = 2 };
struct Job {
    int kind, seq;
};

struct SmemV {
    alignas(128) unsigned char stage[kStagesV][kStageBytes];
    uint64_t full[kStagesV];
    uint64_t empty[kStagesV];
    uint64_t rec_full[kRecs];
    uint64_t rec_empty[kRecs];
    uint64_t work_full[kWork];
    uint64_t work_empty[kWork];
    uint64_t prio_full;   // scheduler -> issuer: one tail task ahead of queued main items
    uint64_t prio_empty;
    uint64_t job_full[kJobs];
    uint64_t job_empty[kJobs];
    Job job[kJobs];
    alignas(16) float2 tsel[kFinishers][kMaxTailChunks * kCW];  // each finisher's copy of one sequence's slice partials
    alignas(16) unsigned char sslice[kFinishers][2][kSliceMax * 2];  // each finisher's chosen slice of p and q
    int job_take;
    Desc desc[kStagesV];
    Work work[kWork];
    Work prio;
    Rec rec[kRecs];
    int n_valid;
    int batch_bad;
    int offs[kSmemSeqs + 1];
    float temp[kSmemSeqs];
    int tok[kSmemToks];
};

template <typename Elem>
__device__ __forceinline__ float load_elem(const void* p) {
    if constexpr (sizeof(Elem) == 2)
        return __uint_as_float(static_cast<uint32_t>(*static_cast<const uint16_t*>(p)) << 16);
    else
        return *static_cast<const float*>(p);
}

// Element e of a staged piece: shared memory first, then the unaligned tail.
template <typename Elem>
__device__ __forceinline__ float piece_elem(const unsigned char* st, int nsm, int skip, const char* tail, int e) {
    return e < nsm ? load_elem<Elem>(st + static_cast<size_t>(e + skip) * sizeof(Elem))
                   : load_elem<Elem>(tail + static_cast<size_t>(e - nsm) * sizeof(Elem));
}

// Residual weight max(0, p - q) of one id, and p itself.
// nz0, nz1: log2 of the normalisers of p and q in the exp2 domain, so that
// p(v) = exp2(x_v c2 - nz0).
__device__ __forceinline__ float resid_w(float xp, float xq, float c2, float nz0, float nz1, float& pv) {
    pv = soft_w(xp, c2, nz0);
    const float qv = soft_w(xq, c2, nz1);
    return fmaxf(0.0f, __fsub_rn(pv, qv));
}

// Softmax partials in the mc domain: (mc, s) holds sum exp2(x c2 - mc);
// merge_mc (isd_device.cuh) merges two of them.
__device__ __forceinline__ void warp_merge_mc(float& M, float& S) {
    const float W = warp_max(M);
    S = (M == -INFINITY) ? 0.0f : S * ex2_approx(M - W);
    S = warp_sum(S);
    M = W;
}

__device__ __forceinline__ void warp_merge_arg(float& M, int& I) {
    const float W = warp_max(M);
    I = warp_min_int(M == W ? I : INT_MAX);
    M = W;
}

// Sequence lookups on a table in shared memory (small batches) or global memory.
__device__ __forceinline__ int seq_of_position_t(const int* offs, int C, int r) {
    int lo = 0, hi = C - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (offs[mid] <= r)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

__device__ __forceinline__ SeqInfo seq_info_t(const int* offs, const float* temp, int i, int total) {
    SeqInfo s;
    s.start = offs[i];
    const int end = offs[i + 1];
    s.len = end - s.start;
    s.T = temp[i];
    s.in_range = s.start >= 0 && end <= total && s.len >= 0;
    s.ok = s.in_range && s.len >= 1 && s.len <= kMaxStride && temperature_ok(s.T);
    return s;
}

__device__ __forceinline__ SeqInfo seq_lookup(const VerifyArgs& a, const SmemV& sm, int i) {
    return a.num_seqs <= kSmemSeqs ? seq_info_t(sm.offs, sm.temp, i, a.total)
                                   : seq_info_t(a.seq_offsets, a.temperature, i, a.total);
}

// ---- outputs of an invalid sequence (one warp) -------------------------------
__device__ void write_invalid(const VerifyArgs& a, int i, const SeqInfo& s, int lane, int code) {
    if (s.in_range) {
        for (int m = lane; m <= s.len; m += 32) a.out_tokens[s.start + i + m] = -1;
        for (int k = lane; k < s.len; k += 32) a.ratio[s.start + k] = NAN;
        if (a.fused)
            for (int k = lane; k < s.len; k += 32) a.proposals[s.start + k] = -1;
    }
    if (lane == 0) {
        a.accept_len[i] = code;
        a.alpha[i] = NAN;
        if (a.fused) a.valid[i] = 0;
    }
}

__device__ __forceinline__ void finalize(const VerifyArgs& a) { atomicAdd(&a.ctl->finalized, 1); }

// ---- pieces of rows for 1-D bulk copies ---------------------------------------
struct Piece {
    uintptr_t lo;
    int bytes, nsm, skip;
    const char* tail;
};

// The 16-byte aligned part of elements [e0, e0 + n) of a row goes to shared
// memory by bulk copy; the unaligned end (fewer than 16 bytes) is read from
// global memory.
template <int E>
__device__ __forceinline__ Piece make_piece(const char* row, int e0, int n) {
    Piece pc;
    const uintptr_t sb = reinterpret_cast<uintptr_t>(row) + static_cast<uintptr_t>(e0) * E;
    const uintptr_t eb = sb + static_cast<uintptr_t>(n) * E;
    const uintptr_t lo = sb & ~static_cast<uintptr_t>(15), hi = eb & ~static_cast<uintptr_t>(15);
    pc.lo = lo;
    if (hi > lo) {
        pc.bytes = static_cast<int>(hi - lo);
        pc.skip = static_cast<int>((sb - lo) / E);
        pc.nsm = static_cast<int>((hi - sb) / E);
    } else {
        pc.bytes = 0;
        pc.skip = 0;
        pc.nsm = 0;
    }
    pc.tail = reinterpret_cast<const char*>(sb) + static_cast<size_t>(pc.nsm) * E;
    return pc;
}

// Slice of a tail sub-chunk of n ids owned by consumer warp w: ids [b, e).
// Slices start on 16-byte boundaries of the sub-chunk.
template <int E>
__device__ __forceinline__ void tail_slice(int n, int w, int& b, int& e) {
    constexpr int vec = 16 / E;
    const int spw = ((n + kCW - 1) / kCW + vec - 1) / vec * vec;
    b = min(n, w * spw);
    e = min(n, b + spw);
}

// =============================================================================
// Bookkeeper warp
// =============================================================================

// Decision of sequence i (L <= 32: lane k handles position k + 1).
template <typename Elem>
__device__ void decide_warp(const VerifyArgs& a, const SmemV& sm, int i, int lane) {
    constexpr int E = sizeof(Elem);
    // The bookkeeper's acquiring count saw every partial of this sequence
    // published; the job ring orders that before this warp's loads.
    const SeqInfo s = seq_lookup(a, sm, i);
    const int L = s.len;
    const float T = s.T;
    const float c2 = T > 0.0f ? inv_temp_log2e(T) : 0.0f;
    const int r = s.start + lane;
    const bool mine = lane < L;
    const int x = mine ? (a.total <= kSmemToks ? sm.tok[r] : __ldg(a.tokens + r)) : 0;
    if (__any_sync(0xffffffffu, mine && (x < 0 || x >= a.vocab))) {
        write_invalid(a, i, s, lane, -1);
        if (lane == 0) {
            a.seq_count[i] = 0;
            finalize(a);
        }
        return;
    }
    float ratio = 0.0f, racc = 0.0f, Mp = -INFINITY, Sp = 0.0f, Mq = -INFINITY, Sq = 0.0f;
    int amax = INT_MAX;
    if (mine) {
        const float2* pp = a.part + static_cast<size_t>(2 * r) * a.nseg;
        const float2* pq = pp + a.nseg;
        // Every load of this lane is issued before any is used.
        float zp = 0.0f, zq = 0.0f;
        if (T > 0.0f) {  // the proposed token's logits, from rows read moments ago
            zp = load_elem<Elem>(a.p + static_cast<int64_t>(r + i) * a.ldp_bytes + static_cast<size_t>(x) * E);
            zq = load_elem<Elem>(a.q + static_cast<int64_t>(r) * a.ldq_bytes + static_cast<size_t>(x) * E);
        }
        float M = -INFINITY;
        for (int j0 = 0; j0 < a.nseg; j0 += 8) {
            float2 u[8], v[8];
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                const int j = j0 + jj;
                u[jj] = j < a.nseg ? __ldcg(pp + j) : make_float2(-INFINITY, 0.0f);
                v[jj] = (T > 0.0f && j < a.nseg) ? __ldcg(pq + j) : make_float2(-INFINITY, 0.0f);
            }
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                if (T > 0.0f) {
                    merge_mc(Mp, Sp, u[jj].x, u[jj].y);
                    merge_mc(Mq, Sq, v[jj].x, v[jj].y);
                } else if (j0 + jj < a.nseg) {
                    merge_argmax(M, amax, u[jj].x, __float_as_int(u[jj].y));
                }
            }
        }
        if (T > 0.0f) {
            const float lp = __fmaf_rn(zp, c2, -Mp) - log2f(Sp);
            const float lq = __fmaf_rn(zq, c2, -Mq) - log2f(Sq);
            ratio = lq == -INFINITY ? 1.0f : fminf(1.0f, exp2f(lp - lq));
            // Relaxed acceptance tests min(1, (1 + tau) p/q); the reported
            // ratio stays the strict one.
            racc = (lq == -INFINITY || a.relax_log2 == 0.0f) ? ratio : fminf(1.0f, exp2f(lp - lq + a.relax_log2));
        } else {
            ratio = x == amax ? 1.0f : 0.0f;
            racc = ratio;
        }
    }
    bool acc = false;
    if (mine) acc = T > 0.0f ? decision_uniform(a.seed, a.offset, i, lane + 1, kTagAccept) < racc : ratio == 1.0f;
    const unsigned bits = __ballot_sync(0xffffffffu, acc);
    const int na = min(bits == 0xffffffffu ? 32 : __ffs(~bits) - 1, L);
    const float total = warp_sum(ratio);
    if (mine) a.ratio[r] = ratio;
    for (int m = lane; m <= L; m += 32) {
        if (m < na) a.out_tokens[s.start + i + m] = x;  // m < na <= 32: m is this lane
        else if (m > na) a.out_tokens[s.start + i + m] = -1;
    }
    const int amax_j = __shfl_sync(0xffffffffu, amax, na & 31);
    const float mc0 = __shfl_sync(0xffffffffu, Mp, na & 31), sp0 = __shfl_sync(0xffffffffu, Sp, na & 31);
    const float mc1 = __shfl_sync(0xffffffffu, Mq, na & 31), sq0 = __shfl_sync(0xffffffffu, Sq, na & 31);
    if (lane == 0) {
        a.accept_len[i] = na;
        a.alpha[i] = total / static_cast<float>(L);
    }
    // The fused call draws the next stride's proposals of a sequence that
    // accepts its whole stride (the others' would be discarded).
    const bool props = a.fused && na == L;
    if (a.fused) {
        if (lane == 0) a.valid[i] = props ? 1 : 0;
        if (!props)
            for (int m = lane; m < L; m += 32) a.proposals[s.start + m] = -1;
    }
    int tok = -1;  // greedy: the token, known now
    if (T == 0.0f) {
        // Greedy: the correction is the argmax of p_j, already known; the
        // bonus is the argmax of p_{L+1}, streamed in the last position's q
        // slot.
        tok = amax_j;
        if (na == L) {
            const float2* pb = a.part + static_cast<size_t>(2 * (s.start + L - 1) + 1) * a.nseg;
            float M = -INFINITY;
            int I = INT_MAX;
            for (int g = lane; g < a.nseg; g += 32) {
                const float2 v = __ldcg(pb + g);
                merge_argmax(M, I, v.x, __float_as_int(v.y));
            }
            warp_merge_arg(M, I);
            tok = I;
        }
        if (lane == 0) a.out_tokens[s.start + i + na] = tok;
    }
    // Tails: the correction or bonus draw (T > 0), then one per proposal row.
    const int n_tok = T > 0.0f ? 1 : 0;
    const int n_pub = n_tok + (props ? L : 0);
    if (n_pub == 0) {
        if (lane == 0) {
            a.seq_count[i] = 0;
            finalize(a);
        }
        return;
    }
    const int mode_tok = na < L ? kTailRes : kTailSoft;
    const int mode_prop = (T > 0.0f ? kTailSoft : kTailArg) | kTailQnew;
    float nz0 = 0.0f, nz1 = 0.0f;
    if (na < L) {
        nz0 = __fadd_rn(mc0, log2f(sp0));
        nz1 = __fadd_rn(mc1, log2f(sq0));
    }
    // Tail record k of this decision (k < n_tok: the token; else proposal
    // row k - n_tok): its tail id and what its producers and selection need.
    auto tail_of = [&](int k, SeqTail& t) -> int {
        t = SeqTail{};
        t.seq = i;
        t.a = na;
        t.c2 = c2;
        if (k < n_tok) {
            t.mode = mode_tok;
            t.prow = s.start + i + na;  // p_j, or p_{L+1} when na == L
            t.qrow = s.start + na;
            t.nz0 = nz0;
            t.nz1 = nz1;
            t.pos = na + 1;
            t.tag = na < L ? kTagCorrect : kTagBonus;
            t.dest = s.start + i + na;
            return i;
        }
        const int row = s.start + (k - n_tok);  // qnew row of position m = k - n_tok + 1
        t.mode = mode_prop;
        t.prow = row;
        t.pos = k - n_tok + 1;
        t.tag = kTagPropose;
        t.dest = -1 - row;
        return a.num_seqs + row;
    };
    int base = 0;
    if (lane == 0) {
        a.seq_pending[i] = n_pub;
        a.seq_count[i] = 0;
        base = atomicAdd(&a.ctl->tail_reserve, n_pub * a.ntask);
    }
    base = __shfl_sync(0xffffffffu, base, 0);
    for (int k = lane; k < n_pub; k += 32) {
        SeqTail t;
        const int id = tail_of(k, t);
        a.tails[id] = t;
    }
    // Every task record carries what its producer needs, so that taking a
    // task is one round trip.
    for (int e = lane; e < n_pub * a.ntask; e += 32) {
        const int k = e / a.ntask, y = e - k * a.ntask;
        SeqTail t;
        const int id = tail_of(k, t);
        int4* tr = a.tasks + 2 * static_cast<size_t>(base + e);
        tr[0] = make_int4(id, y, t.mode, t.prow);
        tr[1] = make_int4(t.qrow, __float_as_int(t.c2), __float_as_int(t.nz0), __float_as_int(t.nz1));
    }
    // Tail state and tasks are visible before any task is flagged ready.
    __threadfence();
    __syncwarp();
    for (int e = lane; e < n_pub * a.ntask; e += 32) st_volatile(a.task_ready + base + e, 1);
}

// Selection of sequence i's token from its tail partials (one warp).  The
// partials are per (tail sub-chunk, consumer warp) slice of about 500 ids;
// the draw picks a slice from them, then scans that slice in vocabulary
// order from registers.
template <typename Elem>
__device__ void select_warp(const VerifyArgs& a, SmemV& sm, int fi, int i, int lane) {
    constexpr int E = sizeof(Elem);
    // One round trip: the tail state (written by the decision before its tasks
    // were published) and every slice partial, into shared memory.
    const int4* tw = reinterpret_cast<const int4*>(a.tails + i);
    int4 tv = make_int4(0, 0, 0, 0);
    if (lane < 3) tv = __ldcg(tw + lane);
    const int U = a.nt * kCW;  // even: 16-byte pairs of partials
    const float4* tp = reinterpret_cast<const float4*>(a.tpart + static_cast<size_t>(i) * U);
    float4* ts = reinterpret_cast<float4*>(sm.tsel[fi]);
    for (int u = lane; u < U / 2; u += 32) cp_async16(ts + u, tp + u);
    cp_async_wait_all();
    SeqTail t;
    const int mode_flags = __shfl_sync(0xffffffffu, tv.x, 0);
    t.mode = mode_flags & ~kTailQnew;
    t.a = __shfl_sync(0xffffffffu, tv.y, 0);
    t.prow = __shfl_sync(0xffffffffu, tv.z, 0);
    t.qrow = __shfl_sync(0xffffffffu, tv.w, 0);
    t.c2 = __int_as_float(__shfl_sync(0xffffffffu, tv.x, 1));
    t.nz0 = __int_as_float(__shfl_sync(0xffffffffu, tv.y, 1));
    t.nz1 = __int_as_float(__shfl_sync(0xffffffffu, tv.z, 1));
    t.seq = __shfl_sync(0xffffffffu, tv.w, 1);
    t.pos = __shfl_sync(0xffffffffu, tv.x, 2);
    t.tag = __shfl_sync(0xffffffffu, tv.y, 2);
    t.dest = __shfl_sync(0xffffffffu, tv.z, 2);
    __syncwarp();
    // The draw is written to its slot; the sequence is final with its last draw.
    auto finish = [&](int token) {
        if (lane == 0) {
            if (t.dest >= 0)
                a.out_tokens[t.dest] = token;
            else
                a.proposals[-1 - t.dest] = token;
            a.tail_count[i] = 0;
            if (atomicSub(a.seq_pending + t.seq, 1) == 1) finalize(a);
        }
    };
    if (t.mode == kTailArg) {  // greedy proposal: merge the slice argmaxes
        float M = -INFINITY;
        int I = INT_MAX;
        for (int u = lane; u < U; u += 32) merge_argmax(M, I, sm.tsel[fi][u].x, __float_as_int(sm.tsel[fi][u].y));
        warp_merge_arg(M, I);
        finish(I);
        return;
    }
    // Slice weights in one scale, the target u * total, and its slice.  Lane
    // l owns the consecutive slices [l * ub, (l + 1) * ub): the lanes reduce
    // their blocks locally and meet in one scan, so the pass costs a handful
    // of shuffles instead of a few per 32 slices.
    const int ub = (U + 31) / 32;
    const int u_lo = min(U, lane * ub), u_hi = min(U, u_lo + ub);
    float MC = -INFINITY, W = 0.0f;
    for (int u = u_lo; u < u_hi; ++u) {
        const float x = sm.tsel[fi][u].x;
        MC = fmaxf(MC, x);
        W += x;
    }
    bool fallback = false;
    if (t.mode == kTailSoft) MC = warp_max(MC);
    else fallback = !(warp_sum(W) > 0.0f);  // residual rounded to zero: draw from p_j
    auto slice_w = [&](int u) -> float {
        const float2 v = sm.tsel[fi][u];
        if (t.mode == kTailSoft) return v.x == -INFINITY ? 0.0f : v.y * ex2_approx(v.x - MC);
        return fallback ? v.y : v.x;
    };
    const float rnd = decision_uniform(a.seed, a.offset, t.seq, t.pos, t.tag);
    float own = 0.0f;
    int lpos = -1;  // the lane's last slice with positive weight
    for (int u = u_lo; u < u_hi; ++u) {
        const float w = slice_w(u);
        own += w;
        if (w > 0.0f) lpos = u;
    }
    float incl = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    const float target = rnd * __shfl_sync(0xffffffffu, incl, 31);
    const unsigned hit = __ballot_sync(0xffffffffu, u_hi > u_lo && incl > target);
    int chosen = -1;
    float tloc = INFINITY;
    if (hit) {
        const int owner = __ffs(hit) - 1;
        if (lane == owner) {  // in-order scan of the owner's block
            float cum = incl - own;
            for (int u = u_lo; u < u_hi; ++u) {
                const float w = slice_w(u);
                if (cum + w > target) {
                    chosen = u;
                    tloc = target - cum;
                    break;
                }
                cum += w;
            }
            if (chosen < 0) chosen = lpos;  // rounding inside the block: its last positive slice
        }
        chosen = __shfl_sync(0xffffffffu, chosen, owner);
        tloc = __shfl_sync(0xffffffffu, tloc, owner);
    }
    if (chosen < 0) {  // rounding left the target past the last weight
        const int last_pos = warp_max_int(lpos);
        chosen = last_pos >= 0 ? last_pos : 0;
        tloc = INFINITY;
    }
    // The chosen slice: ids [lo, lo + len) of the tail row(s).
    const int c = chosen / kCW, w = chosen % kCW;
    const int nc = min(a.ckt, a.vocab - c * a.ckt);
    int sb, se;
    tail_slice<E>(nc, w, sb, se);
    const int lo = c * a.ckt + sb;
    const int len = se - sb;
    const char* prow = (mode_flags & kTailQnew) ? a.qnew + static_cast<int64_t>(t.prow) * a.ldqnew_bytes
                                                : a.p + static_cast<int64_t>(t.prow) * a.ldp_bytes;
    const char* qrow = a.q + static_cast<int64_t>(t.qrow) * a.ldq_bytes;
    constexpr int kVec = 16 / E;
    constexpr int kPer = 2 * kVec;  // ids per lane: at most two 16-byte vectors
    static_assert(kPer * 32 * E == kSliceMax * 2, "a slice fills at most two vectors per lane");
    const int q = ((len + 31) / 32 + kVec - 1) / kVec * kVec;  // whole vectors per lane
    const int b = lane * q;
    const int cnt = max(0, min(q, len - b));
    // Stage the slice's logits in shared memory with every load in flight at
    // once: 16-byte copies where both rows allow them, then the elements
    // left (all of them for rows that are not 16-byte aligned).
    const bool res = t.mode != kTailSoft;
    unsigned char* sp = sm.sslice[fi][0];
    unsigned char* sq = sm.sslice[fi][1];
    const char* gp = prow + static_cast<size_t>(lo) * E;
    const char* gq = qrow + static_cast<size_t>(lo) * E;
    const bool v16 = (reinterpret_cast<uintptr_t>(gp) & 15u) == 0 && (!res || (reinterpret_cast<uintptr_t>(gq) & 15u) == 0);
    const int nv16 = v16 ? (len * E) >> 4 : 0;
    for (int v = lane; v < nv16; v += 32) {
        cp_async16(sp + 16 * v, gp + 16 * v);
        if (res) cp_async16(sq + 16 * v, gq + 16 * v);
    }
    using Raw = typename std::conditional<E == 2, uint16_t, uint32_t>::type;
    for (int e0 = nv16 * (16 / E); e0 < len; e0 += 4 * 32) {
        Raw rp[4], rq[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int e = e0 + lane + 32 * j;
            rp[j] = e < len ? reinterpret_cast<const Raw*>(gp)[e] : Raw(0);
            rq[j] = (res && e < len) ? reinterpret_cast<const Raw*>(gq)[e] : Raw(0);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int e = e0 + lane + 32 * j;
            if (e < len) {
                reinterpret_cast<Raw*>(sp)[e] = rp[j];
                if (res) reinterpret_cast<Raw*>(sq)[e] = rq[j];
            }
        }
    }
    cp_async_wait_all();
    __syncwarp();
    const uint4* sp4 = reinterpret_cast<const uint4*>(sp) + b / kVec;
    const uint4* sq4 = reinterpret_cast<const uint4*>(sq) + b / kVec;
    uint4 P[2], Q[2];
#pragma unroll
    for (int v = 0; v < 2; ++v) {
        P[v] = v * kVec < cnt ? sp4[v] : make_uint4(0, 0, 0, 0);
        Q[v] = (res && v * kVec < cnt) ? sq4[v] : make_uint4(0, 0, 0, 0);
    }
    float wv[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
        wv[k] = 0.0f;
        if (k < cnt) {
            const float xp = vec_elem<E>(P[k / kVec], k % kVec);
            if (!res) {
                wv[k] = soft_w(xp, t.c2, MC);
            } else {
                float pv;
                const float rw = resid_w(xp, vec_elem<E>(Q[k / kVec], k % kVec), t.c2, t.nz0, t.nz1, pv);
                wv[k] = fallback ? pv : rw;
            }
        }
    }
    float own2 = 0.0f;
    int lp = -1;
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
        own2 += wv[k];
        if (wv[k] > 0.0f) lp = b + k;
    }
    float incl2 = own2;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, incl2, o);
        if (lane >= o) incl2 += y;
    }
    const unsigned hit2 = __ballot_sync(0xffffffffu, cnt > 0 && incl2 > tloc);
    int found = -1;
    if (hit2) {
        const int owner = __ffs(hit2) - 1;
        if (lane == owner) {
            float cum = incl2 - own2;
#pragma unroll
            for (int k = 0; k < kPer; ++k) {
                cum += wv[k];
                if (found < 0 && k < cnt && cum > tloc) found = b + k;
            }
            if (found < 0) found = lp;  // rounding inside this lane's ids
        }
        found = __shfl_sync(0xffffffffu, found, owner);
    }
    const int last = warp_max_int(lp);
    finish(lo + (found >= 0 ? found : (last >= 0 ? last : 0)));
}

// Hand a decision or selection to the finisher warp (lane 0 of the bookkeeper).
__device__ __forceinline__ void push_job(const VerifyArgs& a, SmemV& sm, long long& nj, int kind, int seq) {
    const int js = static_cast<int>(nj % kJobs);
    const uint32_t parity = (static_cast<uint32_t>(nj / kJobs) & 1u) ^ 1u;
    ++nj;
    if (!mbar_wait_ns(&sm.job_empty[js], parity, kDrainWaitNs)) atomicOr(&a.ctl->err, kErrWaitTimeout);
    sm.job[js].kind = kind;
    sm.job[js].seq = seq;
    mbar_arrive(&sm.job_full[js]);
}

// Warp reductions within aligned groups of 8 lanes.
__device__ __forceinline__ void group8_merge_mc(float& M, float& S) {
    float W = M;
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) W = fmaxf(W, __shfl_xor_sync(0xffffffffu, W, o, 8));
    S = (M == -INFINITY) ? 0.0f : S * ex2_approx(M - W);
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) S += __shfl_xor_sync(0xffffffffu, S, o, 8);
    M = W;
}
__device__ __forceinline__ void group8_merge_arg(float& M, int& I) {
    float W = M;
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) W = fmaxf(W, __shfl_xor_sync(0xffffffffu, W, o, 8));
    I = M == W ? I : INT_MAX;
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) I = min(I, __shfl_xor_sync(0xffffffffu, I, o, 8));
    M = W;
}

// Records are taken in batches of up to four that are already complete; lane
// group g (8 lanes, one per consumer warp) handles record r + g, so the
// device-scope counts of a batch overlap in one round trip.
__device__ void bookkeeper(const VerifyArgs& a, SmemV& sm, int lane) {
    long long nj = 0;
    const int g = lane >> 3, wl = lane & 7;
    for (long long r = 0;;) {
        // Consumers may idle until other CTAs finish, hence the long bound.
        const bool ok = __all_sync(0xffffffffu, mbar_wait_ns(&sm.rec_full[r % kRecs],
                                                             static_cast<uint32_t>(r / kRecs) & 1u,
                                                             kDrainWaitNs + kWaitNs));
        if (!ok) {
            if (lane == 0) atomicOr(&a.ctl->err, kErrWaitTimeout);
            break;
        }
        int nb = 1;
        while (nb < 4 && mbar_test(&sm.rec_full[(r + nb) % kRecs], static_cast<uint32_t>((r + nb) / kRecs) & 1u))
            ++nb;
        const bool mine = g < nb;
        const Rec& rc = sm.rec[(r + (mine ? g : 0)) % kRecs];
        const int kind = rc.kind, flags = rc.flags, seq = rc.seq, rslot = rc.slot, seg = rc.seg, expect = rc.expect;
        const float2 v = rc.wp[wl];
        __syncwarp();
        if (lane < nb) mbar_arrive(&sm.rec_empty[(r + lane) % kRecs]);
        // An end marker is the last record: the batch stops there.
        const unsigned end_mask = __ballot_sync(0xffffffffu, mine && wl == 0 && kind == kEnd);
        const int n_real = end_mask ? (__ffs(end_mask) - 1) / 8 : nb;
        const bool act = g < n_real;
        int trig = 0;  // 1: decide this sequence, 2: select its token
        // Both merges run on every lane (shuffles need the whole warp); each
        // group keeps the one its record asks for.
        float Mm = v.x, Sm = v.y;
        group8_merge_mc(Mm, Sm);
        float Ma = v.x;
        int Ia = __float_as_int(v.y);
        group8_merge_arg(Ma, Ia);
        // A tail record's eight slice partials, gathered to the group leader so
        // that its releasing count publishes them.
        float2 sl[kCW];
#pragma unroll
        for (int k = 0; k < kCW; ++k) {
            sl[k].x = __shfl_sync(0xffffffffu, v.x, (lane & ~7) + k);
            sl[k].y = __shfl_sync(0xffffffffu, v.y, (lane & ~7) + k);
        }
        if (act && wl == 0) {
            if (kind == kMain) {
                a.part[static_cast<size_t>(rslot) * a.nseg + seg] =
                    flags == kRecArg ? make_float2(Ma, __int_as_float(Ia)) : make_float2(Mm, Sm);
                if (atomic_add_acq_rel(a.seq_count + seq, 1) == expect - 1) trig = 1;
            } else {
                float4* dst = reinterpret_cast<float4*>(a.tpart + (static_cast<size_t>(seq) * a.nt + rslot) * kCW);
#pragma unroll
                for (int k = 0; k < kCW / 2; ++k) dst[k] = make_float4(sl[2 * k].x, sl[2 * k].y, sl[2 * k + 1].x, sl[2 * k + 1].y);
                if ((flags & kLast) && atomic_add_acq_rel(a.tail_count + seq, 1) == a.ntask - 1) trig = 2;
            }
        }
        // Hand the triggered jobs to the finishers, in record order.
        const unsigned tmask = __ballot_sync(0xffffffffu, trig != 0);
        for (unsigned m = tmask; m; m &= m - 1) {
            const int src = __ffs(m) - 1;
            const int tk = __shfl_sync(0xffffffffu, trig, src), ts = __shfl_sync(0xffffffffu, seq, src);
            if (lane == 0) push_job(a, sm, nj, tk == 1 ? kJobDecide : kJobSelect, ts);
        }
        __syncwarp();
        r += nb;
        if (end_mask) break;
    }
    if (lane == 0)
        for (int f = 0; f < kFinishers; ++f) push_job(a, sm, nj, kJobEnd, 0);
}

template <typename Elem>
__device__ void finisher(const VerifyArgs& a, SmemV& sm, int fi, int lane) {
    for (;;) {
        // Jobs are claimed in order by whichever finisher is free.
        int j = 0;
        if (lane == 0) j = atomicAdd(&sm.job_take, 1);
        j = __shfl_sync(0xffffffffu, j, 0);
        const int js = j % kJobs;
        const uint32_t parity = static_cast<uint32_t>(j / kJobs) & 1u;
        const bool ok = __all_sync(0xffffffffu, mbar_wait_ns(&sm.job_full[js], parity, kDrainWaitNs + 2 * kWaitNs));
        if (!ok) {
            if (lane == 0) atomicOr(&a.ctl->err, kErrWaitTimeout);
            return;
        }
        const int kind = sm.job[js].kind, seq = sm.job[js].seq;
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.job_empty[js]);
        if (kind == kJobEnd) return;
        if (kind == kJobDecide)
            decide_warp<Elem>(a, sm, seq, lane);
        else
            select_warp<Elem>(a, sm, fi, seq, lane);
    }
}

// =============================================================================
// Scheduler thread: decides what to stream next, absorbing every global
// memory round trip (work counter, ticket flags, task records, sequence
// lookups) so that the issuer never waits on one.
// =============================================================================

struct SeqCache {
    int i, start, end, len;
    float T;
    bool ok;
};

// Main item w as work for the issuer; false if the item reads nothing.
__device__ bool main_work(const VerifyArgs& a, const SmemV& sm, long long w, SeqCache& sc, Work& wk) {
    const int slot = static_cast<int>(w / a.nseg);
    const int seg = static_cast<int>(w - static_cast<long long>(slot) * a.nseg);
    const int r = slot >> 1, kind = slot & 1;
    if (!(r >= sc.start && r < sc.end)) {
        const bool small = a.num_seqs <= kSmemSeqs;
        const int* offs = small ? sm.offs : a.seq_offsets;
        const int i = seq_of_position_t(offs, a.num_seqs, r);
        const SeqInfo s = seq_lookup(a, sm, i);
        sc.i = i;
        sc.start = s.start;
        sc.len = s.len;
        sc.end = s.in_range ? s.start + max(s.len, 0) : s.start;
        sc.T = s.T;
        sc.ok = s.ok;
        if (!(r >= sc.start && r < sc.end)) {
            sc.start = sc.end = 0;
            return false;  // position outside every sequence
        }
    }
    if (!sc.ok) return false;
    // Greedy verification reads no q rows; the last position's q slot streams
    // the final anchor row p_{L+1} instead, whose argmax is the bonus token.
    const bool greedy = !(sc.T > 0.0f);
    const bool bonus = greedy && kind == 1;
    if (bonus && r != sc.start + sc.len - 1) return false;
    wk.kind = kMain;
    wk.seq = sc.i;
    wk.slot = slot;
    wk.seg = seg;
    wk.expect = (greedy ? sc.len + 1 : 2 * sc.len) * a.nseg;
    // A rejection is likeliest at the first position: its rows stay in L2
    // for the residual tail when the batch can afford it.
    wk.keep = a.keep_first && !greedy && r == sc.start;
    wk.c0 = seg * a.spseg;
    wk.c1 = min(wk.c0 + a.spseg, a.nck);
    wk.c2 = sc.T > 0.0f ? inv_temp_log2e(sc.T) : 0.0f;
    wk.row0 = bonus  ? a.p + static_cast<int64_t>(r + sc.i + 1) * a.ldp_bytes
              : kind ? a.q + static_cast<int64_t>(r) * a.ldq_bytes
                     : a.p + static_cast<int64_t>(r + sc.i) * a.ldp_bytes;
    wk.row1 = nullptr;
    return true;
}

// Tail task of a published queue slot as work for the issuer.
__device__ void tail_work(const VerifyArgs& a, int slot, Work& wk) {
    st_volatile(a.task_ready + slot, 0);
    const int4 w0 = __ldcg(a.tasks + 2 * static_cast<size_t>(slot)), w1 = __ldcg(a.tasks + 2 * static_cast<size_t>(slot) + 1);
    const int i = w0.x, y = w0.y;
    wk.kind = w0.z & ~kTailQnew;
    wk.seq = i;
    wk.slot = 0;
    wk.seg = 0;
    wk.expect = 0;
    wk.keep = 0;
    wk.c0 = y * a.tpt;
    wk.c1 = min(wk.c0 + a.tpt, a.nt);
    wk.c2 = __int_as_float(w1.y);
    wk.nz0 = __int_as_float(w1.z);
    wk.nz1 = __int_as_float(w1.w);
    wk.row0 = (w0.z & kTailQnew) ? a.qnew + static_cast<int64_t>(w0.w) * a.ldqnew_bytes
                                 : a.p + static_cast<int64_t>(w0.w) * a.ldp_bytes;
    wk.row1 = a.q + static_cast<int64_t>(w1.x) * a.ldq_bytes;
}

__device__ void scheduler(const VerifyArgs& a, SmemV& sm, unsigned long long next) {
    bool main_done = sm.batch_bad != 0 || a.n_main == 0;
    SeqCache sc = {0, 0, 0, 0, 0.0f, false};
    // Tail tasks are handed out as tickets: every scheduler holds at most one
    // ticket (a task-queue slot, one atomic to take it) and passes that slot's
    // task to the issuer through a priority slot as soon as a decision
    // publishes it, ahead of the main items already queued.  Every global
    // round trip is issued one pass before its result is looked at.
    const int cap = a.n_tail * a.ntask;
    bool tickets_left = cap > 0;
    int ticket = -1, claim = 0, flag = 0;
    bool claim_pending = false, claim_started = false;
    long long k = 0, kp = 0;  // work items and priority items handed over
    uint64_t t_idle = 0;
    while (true) {
        bool progress = false;
        // 1. A published tail task goes to the priority slot.
        if (claim_pending && ticket < 0) {
            claim_pending = false;
            if (claim < cap) {
                ticket = claim;
                flag = 0;
            } else {
                tickets_left = false;
            }
        }
        if (ticket >= 0 && flag != 0 && mbar_test(&sm.prio_empty, (static_cast<uint32_t>(kp) & 1u) ^ 1u)) {
            __threadfence();  // acquire: the task was published before its flag
            tail_work(a, ticket, sm.prio);
            mbar_arrive(&sm.prio_full);
            ++kp;
            ticket = -1;
            flag = 0;
            if (tickets_left) {
                claim = atomicAdd(&a.ctl->tail_claim, 1);
                claim_pending = true;
            }
            progress = true;
        }
        // 2. The next main item, while the work ring has room.
        if (!main_done) {
            const int ws = static_cast<int>(k % kWork);
            if (mbar_test(&sm.work_empty[ws], (static_cast<uint32_t>(k / kWork) & 1u) ^ 1u)) {
                Work& wk = sm.work[ws];
                bool have = false;
                while (!have && !main_done) {
                    const unsigned long long w = next;
                    if (w < static_cast<unsigned long long>(a.n_main)) {
                        next = atomicAdd(&a.ctl->grab, 1ull);
                        have = main_work(a, sm, static_cast<long long>(w), sc, wk);
                    } else {
                        main_done = true;
                    }
                }
                if (have) {
                    mbar_arrive(&sm.work_full[ws]);
                    ++k;
                    progress = true;
                }
                // The first ticket is claimed once the first main item is on its way.
                if (!claim_started && tickets_left) {
                    claim_started = true;
                    claim = atomicAdd(&a.ctl->tail_claim, 1);
                    claim_pending = true;
                }
            }
        }
        // 3. Refresh the held ticket's flag (looked at on the next pass).
        if (ticket >= 0) flag = ld_volatile(a.task_ready + ticket);
        if (!claim_started && main_done && tickets_left) {
            claim_started = true;
            claim = atomicAdd(&a.ctl->tail_claim, 1);
            claim_pending = true;
        }
        if (progress) {
            t_idle = 0;
            continue;
        }
        if (main_done && ld_volatile(&a.ctl->finalized) >= sm.n_valid) break;  // every sequence is final
        if (t_idle == 0) {
            t_idle = global_timer_ns();
        } else if (global_timer_ns() - t_idle > kDrainWaitNs) {
            atomicOr(&a.ctl->err, kErrWaitTimeout);
            break;
        }
        if (!main_done)  // work ring full: sleep until a slot frees (or ~1 us, to look at the ticket)
            (void)mbar_try_wait_for(&sm.work_empty[k % kWork], (static_cast<uint32_t>(k / kWork) & 1u) ^ 1u, 1000);
        else
            __nanosleep(200);
    }
    // Stop the issuer: an end marker in the work ring (bounded wait for room).
    const int ws = static_cast<int>(k % kWork);
    if (!mbar_wait_ns(&sm.work_empty[ws], (static_cast<uint32_t>(k / kWork) & 1u) ^ 1u, kWaitNs)) {
        atomicOr(&a.ctl->err, kErrWaitTimeout);
        return;
    }
    sm.work[ws].kind = kEnd;
    mbar_arrive(&sm.work_full[ws]);
}

// =============================================================================
// Issuer thread: streams the scheduled work's sub-chunks into the stage ring.
// =============================================================================

__device__ __forceinline__ int acquire_stage(SmemV& sm, long long n, int* err) {
    const int stage = static_cast<int>(n % kStagesV);
    const uint32_t parity = (static_cast<uint32_t>(n / kStagesV) & 1u) ^ 1u;
    if (!mbar_wait_ns(&sm.empty[stage], parity, kWaitNs)) {
        atomicOr(err, kErrWaitTimeout);
        return -1;
    }
    return stage;
}

// Stream sub-chunks [c0, c1) of one unit of work into the stage ring.
template <typename Elem>
__device__ bool issue_work(const VerifyArgs& a, SmemV& sm, const Work& wk, int c0, int c1, long long& n,
                           uint64_t pol_first, uint64_t pol_last) {
    constexpr int E = sizeof(Elem);
    const bool main = wk.kind == kMain;
    const int ck = main ? a.ck : a.ckt;
    for (int c = c0; c < c1; ++c) {
        const int e0 = c * ck;
        const int nel = min(ck, a.vocab - e0);
        const Piece pa = make_piece<E>(wk.row0, e0, nel);
        Piece pb = {};
        if (wk.kind == kTailRes) pb = make_piece<E>(wk.row1, e0, nel);
        const int stage = acquire_stage(sm, n, &a.ctl->err);
        if (stage < 0) return false;
        Desc& d = sm.desc[stage];
        d.kind = wk.kind;
        d.flags = main ? ((c == wk.c0 ? kFirst : 0) | (c == wk.c1 - 1 ? kLast : 0)) : (c == wk.c1 - 1 ? kLast : 0);
        d.seq = wk.seq;
        d.slot = main ? wk.slot : c;
        d.seg = wk.seg;
        d.expect = wk.expect;
        d.e0 = e0;
        d.n = nel;
        d.nvec = pa.bytes >> 4;
        d.nsm0 = pa.nsm;
        d.skip0 = pa.skip;
        d.tail0 = pa.tail;
        d.nsm1 = pb.nsm;
        d.skip1 = pb.skip;
        d.tail1 = pb.tail;
        d.c2 = wk.c2;
        d.nz0 = wk.nz0;
        d.nz1 = wk.nz1;
        const int bytes = pa.bytes + pb.bytes;
        if (bytes > 0) {
            mbar_arrive_expect_tx(&sm.full[stage], static_cast<uint32_t>(bytes));
            const uint64_t pol = wk.keep ? pol_last : pol_first;
            if (pa.bytes > 0)
                bulk_copy_g2s_hint(sm.stage[stage], reinterpret_cast<const void*>(pa.lo),
                                   static_cast<uint32_t>(pa.bytes), &sm.full[stage], pol);
            if (pb.bytes > 0)
                bulk_copy_g2s_hint(sm.stage[stage] + kHalf, reinterpret_cast<const void*>(pb.lo),
                                   static_cast<uint32_t>(pb.bytes), &sm.full[stage], pol);
        } else {
            mbar_arrive(&sm.full[stage]);
        }
        ++n;
    }
    return true;
}

template <typename Elem>
__device__ void issuer(const VerifyArgs& a, SmemV& sm) {
    long long n = 0, kp = 0;
    bool ok = true;
    const uint64_t pol_first = l2_policy_evict_first(), pol_last = l2_policy_evict_last();
    // Tail work waiting in the priority slot goes first, between any two
    // stages; returns -1 on a timeout, 1 if it issued work, 0 otherwise.
    auto priority = [&]() -> int {
        if (!mbar_test(&sm.prio_full, static_cast<uint32_t>(kp) & 1u)) return 0;
        const Work pw = sm.prio;
        mbar_arrive(&sm.prio_empty);
        ++kp;
        return issue_work<Elem>(a, sm, pw, pw.c0, pw.c1, n, pol_first, pol_last) ? 1 : -1;
    };
    for (long long k = 0; ok; ++k) {
        const int ws = static_cast<int>(k % kWork);
        const uint32_t parity = static_cast<uint32_t>(k / kWork) & 1u;
        // Wait for the next main item, serving the priority slot meanwhile.
        const uint64_t t0 = global_timer_ns();
        bool got = false;
        while (ok && !(got = mbar_test(&sm.work_full[ws], parity))) {
            const int pr = priority();
            ok = pr >= 0;
            if (global_timer_ns() - t0 > kDrainWaitNs + kWaitNs) {
                atomicOr(&a.ctl->err, kErrWaitTimeout);
                ok = false;
            }
            if (pr == 0) __nanosleep(200);
        }
        if (!got) break;
        const Work wk = sm.work[ws];
        mbar_arrive(&sm.work_empty[ws]);
        if (wk.kind == kEnd) break;
        for (int c = wk.c0; c < wk.c1 && ok; ++c) {
            ok = priority() >= 0;
            if (ok) ok = issue_work<Elem>(a, sm, wk, c, c + 1, n, pol_first, pol_last);
        }
    }
    const int stage = acquire_stage(sm, n, &a.ctl->err);
    if (stage >= 0) {
        sm.desc[stage].kind = kEnd;
        mbar_arrive(&sm.full[stage]);
    }
}

// =============================================================================
// Consumer warps
// =============================================================================

struct MainState {
    float m, mc;
    uint64_t acc0, acc1;
    int amx;
};

// Hand this warp's partial for the current record to the bookkeeper.
__device__ __forceinline__ void push_record(const VerifyArgs& a, SmemV& sm, long long& nrec, int warp, int lane,
                                            float2 part, int kind, int flags, int seq, int slot, int seg,
                                            int expect) {
    const int rs = static_cast<int>(nrec % kRecs);
    const uint32_t parity = (static_cast<uint32_t>(nrec / kRecs) & 1u) ^ 1u;
    ++nrec;
    if (lane == 0) {
        if (!mbar_wait_ns(&sm.rec_empty[rs], parity, kDrainWaitNs)) atomicOr(&a.ctl->err, kErrWaitTimeout);
        Rec& rc = sm.rec[rs];
        rc.wp[warp] = part;
        if (warp == 0) {
            rc.kind = kind;
            rc.flags = flags;
            rc.seq = seq;
            rc.slot = slot;
            rc.seg = seg;
            rc.expect = expect;
        }
        mbar_arrive(&sm.rec_full[rs]);
    }
    __syncwarp();
}

template <typename Elem>
__device__ __forceinline__ void main_stage(const VerifyArgs& a, SmemV& sm, int stage, const Desc& d, int tid,
                                           int warp, int lane, MainState& ms, long long& nrec) {
    constexpr bool kBf16 = sizeof(Elem) == 2;
    constexpr uint32_t kNeg = kBf16 ? 0xff80ff80u : 0xff800000u;  // -inf pattern
    uint32_t w[kVecPT * 4];
    const uint4* sv = reinterpret_cast<const uint4*>(sm.stage[stage]);
#pragma unroll
    for (int k = 0; k < kVecPT; ++k) {
        const int vi = tid + k * kCT;
        const uint4 v = vi < d.nvec ? sv[vi] : make_uint4(kNeg, kNeg, kNeg, kNeg);
        w[4 * k] = v.x;
        w[4 * k + 1] = v.y;
        w[4 * k + 2] = v.z;
        w[4 * k + 3] = v.w;
    }
    if (d.skip0 != 0 && tid == 0) {  // elements before the sub-chunk in the first vector
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if constexpr (kBf16) {
                if (2 * j < d.skip0) w[j] = (w[j] & 0xffff0000u) | 0xff80u;
                if (2 * j + 1 < d.skip0) w[j] = (w[j] & 0x0000ffffu) | 0xff800000u;
            } else {
                if (j < d.skip0) w[j] = kNeg;
            }
        }
    }
    const int ntail = d.n - d.nsm0;
    float tv = -INFINITY;
    if (tid < ntail) tv = load_elem<Elem>(d.tail0 + static_cast<size_t>(tid) * sizeof(Elem));
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.empty[stage]);

    if (d.flags & kFirst) {
        ms.m = -INFINITY;
        ms.mc = -INFINITY;
        ms.acc0 = 0;
        ms.acc1 = 0;
        ms.amx = INT_MAX;
    }
    float cm;
    if constexpr (kBf16) {
        uint32_t mx = w[0];
#pragma unroll
        for (int j = 1; j < kVecPT * 4; ++j) mx = hmax2_bf16(mx, w[j]);
        cm = fmaxf(bf16lo(mx), bf16hi(mx));
    } else {
        cm = __uint_as_float(w[0]);
#pragma unroll
        for (int j = 1; j < kVecPT * 4; ++j) cm = fmaxf(cm, __uint_as_float(w[j]));
    }
    cm = fmaxf(cm, tv);
    const float c2 = d.c2;
    if (c2 > 0.0f) {
        if (cm > ms.m) {
            const float mcn = cm * c2;
            if (ms.m != -INFINITY) {
                const float sc = ex2_approx(ms.mc - mcn);
                const uint64_t sc2 = pack_f2(sc, sc);
                ms.acc0 = mul_f2(ms.acc0, sc2);
                ms.acc1 = mul_f2(ms.acc1, sc2);
            }
            ms.m = cm;
            ms.mc = mcn;
        }
        if (ms.m != -INFINITY) {
            const uint64_t C2 = pack_f2(c2, c2), NMC = pack_f2(-ms.mc, -ms.mc);
#pragma unroll
            for (int j = 0; j < kVecPT * 4; j += 2) {
                if constexpr (kBf16) {
                    float y0, y1, y2, y3;
                    unpack_f2(fma_f2(pack_f2(bf16lo(w[j]), bf16hi(w[j])), C2, NMC), y0, y1);
                    unpack_f2(fma_f2(pack_f2(bf16lo(w[j + 1]), bf16hi(w[j + 1])), C2, NMC), y2, y3);
                    ms.acc0 = add_f2(ms.acc0, pack_f2(ex2_approx(y0), ex2_approx(y1)));
                    ms.acc1 = add_f2(ms.acc1, pack_f2(ex2_approx(y2), ex2_approx(y3)));
                } else {
                    float y0, y1;
                    unpack_f2(fma_f2(pack_f2(__uint_as_float(w[j]), __uint_as_float(w[j + 1])), C2, NMC), y0, y1);
                    if (j & 2)
                        ms.acc1 = add_f2(ms.acc1, pack_f2(ex2_approx(y0), ex2_approx(y1)));
                    else
                        ms.acc0 = add_f2(ms.acc0, pack_f2(ex2_approx(y0), ex2_approx(y1)));
                }
            }
            if (tv != -INFINITY) ms.acc1 = add_f2(ms.acc1, pack_f2(soft_w(tv, c2, ms.mc), 0.0f));
        }
    } else if (cm > ms.m) {
        // First position of the new maximum in this thread's (ascending) elements.
        constexpr int kPer = kBf16 ? 8 : 4;
        int idx = INT_MAX;
        if (tv == cm) idx = d.nsm0 + tid;
#pragma unroll
        for (int k = kVecPT - 1; k >= 0; --k) {
#pragma unroll
            for (int j = 3; j >= 0; --j) {
                const uint32_t x = w[4 * k + j];
                const int base = (tid + k * kCT) * kPer - d.skip0;
                if constexpr (kBf16) {
                    if (bf16hi(x) == cm) idx = base + 2 * j + 1;
                    if (bf16lo(x) == cm) idx = base + 2 * j;
                } else {
                    if (__uint_as_float(x) == cm) idx = base + j;
                }
            }
        }
        ms.m = cm;
        ms.amx = d.e0 + idx;
    }

    if (d.flags & kLast) {
        float2 part;
        int mode;
        if (c2 > 0.0f) {
            float s0, s1, s2, s3;
            unpack_f2(ms.acc0, s0, s1);
            unpack_f2(ms.acc1, s2, s3);
            float M = ms.m == -INFINITY ? -INFINITY : ms.mc, S = (s0 + s1) + (s2 + s3);
            warp_merge_mc(M, S);
            part = make_float2(M, S);
            mode = kRecSoft;
        } else {
            float M = ms.m;
            int I = ms.amx;
            warp_merge_arg(M, I);
            part = make_float2(M, __int_as_float(I));
            mode = kRecArg;
        }
        push_record(a, sm, nrec, warp, lane, part, kMain, mode, d.seq, d.slot, d.seg, d.expect);
    }
}

// Residual weights of two ids from packed p and q logits: accumulates the
// residual sum and the p sum (bit-identical to resid_w per id).
__device__ __forceinline__ void resid_pair(float xp0, float xp1, float xq0, float xq1, uint64_t C2, uint64_t NZ0,
                                           uint64_t NZ1, uint64_t& sw, uint64_t& sp) {
    float a0, a1, b0, b1;
    unpack_f2(fma_f2(pack_f2(xp0, xp1), C2, NZ0), a0, a1);
    unpack_f2(fma_f2(pack_f2(xq0, xq1), C2, NZ1), b0, b1);
    const uint64_t pv = pack_f2(ex2_approx(a0), ex2_approx(a1));
    const uint64_t qv = pack_f2(ex2_approx(b0), ex2_approx(b1));
    float d0, d1;
    unpack_f2(fma_f2(qv, pack_f2(-1.0f, -1.0f), pv), d0, d1);  // pv - qv, one rounding
    sw = add_f2(sw, pack_f2(fmaxf(0.0f, d0), fmaxf(0.0f, d1)));
    sp = add_f2(sp, pv);
}

// Residual weights of one 16-byte vector of p logits and the matching vector
// of q logits.
template <int E>
__device__ __forceinline__ void resid_vec(const uint4& A, const uint4& B, uint64_t C2, uint64_t NZ0, uint64_t NZ1,
                                          uint64_t& sw, uint64_t& sp) {
    if constexpr (E == 2) {
        resid_pair(bf16lo(A.x), bf16hi(A.x), bf16lo(B.x), bf16hi(B.x), C2, NZ0, NZ1, sw, sp);
        resid_pair(bf16lo(A.y), bf16hi(A.y), bf16lo(B.y), bf16hi(B.y), C2, NZ0, NZ1, sw, sp);
        resid_pair(bf16lo(A.z), bf16hi(A.z), bf16lo(B.z), bf16hi(B.z), C2, NZ0, NZ1, sw, sp);
        resid_pair(bf16lo(A.w), bf16hi(A.w), bf16lo(B.w), bf16hi(B.w), C2, NZ0, NZ1, sw, sp);
    } else {
        resid_pair(__uint_as_float(A.x), __uint_as_float(A.y), __uint_as_float(B.x), __uint_as_float(B.y), C2, NZ0,
                   NZ1, sw, sp);
        resid_pair(__uint_as_float(A.z), __uint_as_float(A.w), __uint_as_float(B.z), __uint_as_float(B.w), C2, NZ0,
                   NZ1, sw, sp);
    }
}

// A tail stage: each consumer warp reduces its own contiguous slice of the
// sub-chunk (about 1/8 of it), so the selection can later narrow a draw down
// to one slice.  A slice holds at most 64 vectors: every lane loads its (at
// most two) vectors of each row up front, then reduces them from registers.
template <typename Elem>
__device__ __forceinline__ void tail_stage(const VerifyArgs& a, SmemV& sm, int stage, const Desc& d, int warp,
                                           int lane, long long& nrec) {
    constexpr int E = sizeof(Elem);
    constexpr int kVec = 16 / E;
    constexpr uint32_t kNeg = E == 2 ? 0xff80ff80u : 0xff800000u;  // -inf pattern
    const unsigned char* s0 = sm.stage[stage];
    const unsigned char* s1 = s0 + kHalf;
    int wb, we;
    tail_slice<E>(d.n, warp, wb, we);
    const bool vec0 = d.skip0 == 0 && d.nsm0 == d.n;  // piece whole and aligned in shared memory
    const bool vec = vec0 && (d.kind != kTailRes || (d.skip1 == 0 && d.nsm1 == d.n));
    // The lane's vectors v, v + 32 of the slice, -inf where past its end.
    const int vb = wb / kVec, ve = we / kVec;
    const int v0 = vb + lane, v1 = v0 + 32;
    const uint4 neg = make_uint4(kNeg, kNeg, kNeg, kNeg);
    uint4 A0 = neg, A1 = neg, B0 = neg, B1 = neg;
    if (vec) {
        const uint4* p4 = reinterpret_cast<const uint4*>(s0);
        if (v0 < ve) A0 = p4[v0];
        if (v1 < ve) A1 = p4[v1];
        if (d.kind == kTailRes) {
            const uint4* q4 = reinterpret_cast<const uint4*>(s1);
            if (v0 < ve) B0 = q4[v0];
            if (v1 < ve) B1 = q4[v1];
        }
    }
    float2 part;
    if (d.kind == kTailRes) {
        float sws = 0.0f, sps = 0.0f;
        if (vec) {
            const uint64_t C2 = pack_f2(d.c2, d.c2);
            const uint64_t NZ0 = pack_f2(-d.nz0, -d.nz0), NZ1 = pack_f2(-d.nz1, -d.nz1);
            uint64_t sw0 = 0, sp0 = 0, sw1 = 0, sp1 = 0;
            resid_vec<E>(A0, B0, C2, NZ0, NZ1, sw0, sp0);
            resid_vec<E>(A1, B1, C2, NZ0, NZ1, sw1, sp1);
            float w0, w1, w2, w3, p0, p1, p2, p3;
            unpack_f2(sw0, w0, w1);
            unpack_f2(sw1, w2, w3);
            unpack_f2(sp0, p0, p1);
            unpack_f2(sp1, p2, p3);
            sws = (w0 + w1) + (w2 + w3);
            sps = (p0 + p1) + (p2 + p3);
        } else {
            for (int e = wb + lane; e < we; e += 32) {
                const float xp = piece_elem<Elem>(s0, d.nsm0, d.skip0, d.tail0, e);
                const float xq = piece_elem<Elem>(s1, d.nsm1, d.skip1, d.tail1, e);
                float pv;
                sws += resid_w(xp, xq, d.c2, d.nz0, d.nz1, pv);
                sps += pv;
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty[stage]);
        part = make_float2(warp_sum(sws), warp_sum(sps));
    } else if (d.kind == kTailSoft) {
        float mt = -INFINITY, st = 0.0f;
        if (vec) {
            mt = fmaxf(vec_max<E>(A0), vec_max<E>(A1));
            if (mt != -INFINITY) {
                const float mct = mt * d.c2;
                const uint64_t C2 = pack_f2(d.c2, d.c2), NMC = pack_f2(-mct, -mct);
                uint64_t acc0 = 0, acc1 = 0;
                soft_vec<E>(A0, C2, NMC, acc0);
                soft_vec<E>(A1, C2, NMC, acc1);
                float a0, a1, a2, a3;
                unpack_f2(acc0, a0, a1);
                unpack_f2(acc1, a2, a3);
                st = (a0 + a1) + (a2 + a3);
            }
        } else {
            for (int e = wb + lane; e < we; e += 32) mt = fmaxf(mt, piece_elem<Elem>(s0, d.nsm0, d.skip0, d.tail0, e));
            if (mt != -INFINITY)
                for (int e = wb + lane; e < we; e += 32)
                    st += soft_w(piece_elem<Elem>(s0, d.nsm0, d.skip0, d.tail0, e), d.c2, mt * d.c2);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty[stage]);
        float M = mt == -INFINITY ? -INFINITY : mt * d.c2, S = st;
        warp_merge_mc(M, S);
        part = make_float2(M, S);
    } else {  // kTailArg: the lane's first maximum in id order
        float mt = -INFINITY;
        int it = INT_MAX;
        if (vec) {
#pragma unroll
            for (int j = 0; j < kVec; ++j) {
                const float x = vec_elem<E>(A0, j);
                if (v0 < ve && x > mt) {
                    mt = x;
                    it = d.e0 + v0 * kVec + j;
                }
            }
#pragma unroll
            for (int j = 0; j < kVec; ++j) {
                const float x = vec_elem<E>(A1, j);
                if (v1 < ve && x > mt) {
                    mt = x;
                    it = d.e0 + v1 * kVec + j;
                }
            }
        } else {
            for (int e = wb + lane; e < we; e += 32) {
                const float x = piece_elem<Elem>(s0, d.nsm0, d.skip0, d.tail0, e);
                if (x > mt) {
                    mt = x;
                    it = d.e0 + e;
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty[stage]);
        warp_merge_arg(mt, it);
        part = make_float2(mt, __int_as_float(it));
    }
    push_record(a, sm, nrec, warp, lane, part, d.kind, d.flags, d.seq, d.slot, 0, 0);
}

template <typename Elem>
__device__ void consumer(const VerifyArgs& a, SmemV& sm, int tid, int warp, int lane) {
    MainState ms = {-INFINITY, -INFINITY, 0, 0, INT_MAX};
    long long nrec = 0;
    long long n = 0;
    for (;; ++n) {
        const int stage = static_cast<int>(n % kStagesV);
        const uint32_t parity = static_cast<uint32_t>(n / kStagesV) & 1u;
        // The issuer may idle until other CTAs finish, hence the long bound.
        if (!__all_sync(0xffffffffu, mbar_wait_ns(&sm.full[stage], parity, kDrainWaitNs + kWaitNs))) {
            if (lane == 0) atomicOr(&a.ctl->err, kErrWaitTimeout);
            break;
        }
        const Desc d = sm.desc[stage];
        if (d.kind == kEnd) break;
        if (d.kind == kMain)
            main_stage<Elem>(a, sm, stage, d, tid, warp, lane, ms, nrec);
        else
            tail_stage<Elem>(a, sm, stage, d, warp, lane, nrec);
    }
    // Tell the bookkeeper there is no more work (a record of kind kEnd).
    push_record(a, sm, nrec, warp, lane, make_float2(0.0f, 0.0f), kEnd, 0, 0, 0, 0, 0);
}

// =============================================================================
// Kernel
// =============================================================================

template <typename Elem>
__global__ void __launch_bounds__(kThreadsV, kVerifyCtasPerSm) verify_kernel(const VerifyArgs a) {
    extern __shared__ unsigned char smem_raw[];
    SmemV& sm = *reinterpret_cast<SmemV*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~static_cast<uintptr_t>(127));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    pdl_wait();
    pdl_launch_dependents();
    if (tid == 0) {
        for (int s = 0; s < kStagesV; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], kCW);
        }
        for (int s = 0; s < kRecs; ++s) {
            mbar_init(&sm.rec_full[s], kCW);
            mbar_init(&sm.rec_empty[s], 1);
        }
        for (int s = 0; s < kWork; ++s) {
            mbar_init(&sm.work_full[s], 1);
            mbar_init(&sm.work_empty[s], 1);
        }
        mbar_init(&sm.prio_full, 1);
        mbar_init(&sm.prio_empty, 1);
        for (int s = 0; s < kJobs; ++s) {
            mbar_init(&sm.job_full[s], 1);
            mbar_init(&sm.job_empty[s], 1);
        }
        fence_mbarrier_init();
        sm.n_valid = 0;
        sm.job_take = 0;
    }
    // The scheduler's first main item, requested while the prologue runs.
    unsigned long long first = 0;
    if (tid == kSchedWarp * 32 && a.n_main > 0) first = atomicAdd(&a.ctl->grab, 1ull);
    // Every CTA counts the valid sequences (the grid's exit condition) and
    // checks that the offsets never decrease; small batches keep the offsets
    // and temperatures in shared memory.
    int nv = 0;
    bool bad = false;
    const bool small = a.num_seqs <= kSmemSeqs;
    for (int i = tid; i < a.num_seqs; i += kThreadsV) {
        const SeqInfo s = seq_info(a.seq_offsets, a.temperature, i, a.total);
        nv += s.ok ? 1 : 0;
        const int end = __ldg(a.seq_offsets + i + 1);
        bad = bad || end < s.start;
        if (small) {
            sm.offs[i] = s.start;
            sm.temp[i] = s.T;
            if (i == a.num_seqs - 1) sm.offs[i + 1] = end;
        }
    }
    if (a.total <= kSmemToks)  // the decisions read the proposed tokens from here
        for (int r = tid; r < a.total; r += kThreadsV) sm.tok[r] = __ldg(a.tokens + r);
    __syncthreads();
    if (nv) atomicAdd(&sm.n_valid, nv);
    bad = __syncthreads_or(bad);
    if (tid == 0) {
        sm.batch_bad = bad;
        if (bad) sm.n_valid = 0;
    }
    __syncthreads();

    if (warp == kIssuerWarp) {
        if (lane == 0) issuer<Elem>(a, sm);
    } else if (warp == kSchedWarp) {
        if (lane == 0) scheduler(a, sm, first);
    } else if (warp == kBookWarp) {
        bookkeeper(a, sm, lane);
    } else if (warp >= kFinWarp) {
        finisher<Elem>(a, sm, warp - kFinWarp, lane);
    } else {
        // This CTA's share of the sequences that are invalid as laid out.
        for (long long i = blockIdx.x + static_cast<long long>(warp) * gridDim.x; i < a.num_seqs;
             i += static_cast<long long>(kCW) * gridDim.x) {
            const SeqInfo s = seq_info(a.seq_offsets, a.temperature, static_cast<int>(i), a.total);
            if (bad || !s.ok) write_invalid(a, static_cast<int>(i), s, lane, -1);
        }
        consumer<Elem>(a, sm, tid, warp, lane);
    }
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        if (atomicAdd(&a.ctl->exited, 1) == static_cast<int>(gridDim.x) - 1) {
            __threadfence();
            if (ld_volatile(&a.ctl->err) != 0)
                for (int i = 0; i < a.num_seqs; ++i) {
                    a.accept_len[i] = -2;
                    if (a.fused) a.valid[i] = 0;
                }
            a.ctl->grab = 0;
            a.ctl->tail_reserve = 0;
            a.ctl->tail_claim = 0;
            a.ctl->finalized = 0;
            a.ctl->exited = 0;
        }
    }
}

static_assert(sizeof(SmemV) + 128 <= 113 * 1024, "two CTAs per SM");

template <typename Elem>
cudaError_t launch_verify_t(const VerifyArgs& a, int grid, cudaStream_t stream) {
    const size_t smem = sizeof(SmemV) + 128;
    cudaError_t err = cudaFuncSetAttribute(verify_kernel<Elem>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreadsV);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, verify_kernel<Elem>, a);
}

}  // namespace

cudaError_t launch_verify(const VerifyArgs& a, int elem_bytes, int grid, cudaStream_t stream) {
    return elem_bytes == 2 ? launch_verify_t<__nv_bfloat16>(a, grid, stream) : launch_verify_t<float>(a, grid, stream);
}

}  // namespace isd
