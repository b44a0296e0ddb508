// The verify step of Introspective Strided Decoding as two kernels
// ("Introspective Diffusion Language Models | Summary", §2 acceptance rate,
// §3.2 strict acceptance, residual correction and bonus token, §3.3 online
// softmax over the vocabulary and a common acceptance path free of
// correction work), optionally with the next stride's proposal draws of the
// fused step (§3.2: one forward verifies and proposes).
//
// stream kernel  every chunk (at most 32 KB) of every row a decision needs:
//                p_k and q_k for k <= L_i (T > 0), or p_1 .. p_{L+1}
//                (T = 0).  Chunks are taken in small batches from a global
//                counter, staged with 1-D bulk copies into a 3-stage ring
//                (mbarrier completion) by one producer thread, and reduced by
//                eight consumer warps to a softmax partial (max, sum) or an
//                argmax per warp; a bookkeeper warp merges the eight, stores
//                the chunk's partial and counts the sequence's chunks, and
//                the CTA that stores a sequence's last chunk publishes its
//                ready word.
// draw kernel    launched behind it (programmatic dependent launch, released
//                as soon as the stream kernel starts): its CTAs run on the
//                SMs the stream leaves room on, then take the SMs as the
//                stream's CTAs retire.  Every warp is a worker:
//                  decisions   by ticket (a sequence index), once the
//                              sequence's ready word is published: ratio_k =
//                              min(1, p_k(x_k) / q_k(x_k)), alpha, the accept
//                              prefix (Philox uniforms, one warp ballot;
//                              relaxed acceptance tests min(1, (1 + tau) p/q))
//                              and the emitted prefix; a greedy correction or
//                              bonus.  The draws left are published as tails;
//                  pieces      by ticket: 4 KB of a tail's row or row pair (the
//                              residual max(0, p_j - q_j) of the one rejected
//                              row pair, the final anchor p_{L+1}, or a qnew
//                              row of the fused call), staged in padded shared
//                              memory and reduced; the weight of every 512-byte
//                              block of the piece is published with the
//                              piece's result;
//                  draws       queued when a tail's last piece is finished and
//                              taken by the workers that run out of pieces:
//                              by inverse CDF (the piece from the piece
//                              weights, the block from its block weights, the
//                              id from the block's logits) or, with the
//                              Gumbel-max sampler, the largest perturbed score.
// Tail descriptors and piece results travel as 64-bit words that carry a
// flag in their high half, so a reader polls the data itself: one global
// round trip per hand-over.  The draw kernel exits once every sequence is
// final; its last CTA re-zeroes the control block.  Every wait is bounded;
// on expiry the error word is set and every accept length reads -2.
#include <climits>
#include <type_traits>

#include "isd_device.cuh"
#include "isd_internal.h"

namespace isd {
namespace {

constexpr int kCW = 8;                 // consumer warps (stream kernel)
constexpr int kCT = kCW * 32;          // consumer threads
constexpr int kProdWarp = kCW;
constexpr int kBookWarp = kCW + 1;
constexpr int kThreadsA = 32 * (kCW + 2);
constexpr int kStagesV = 3;
constexpr int kRecs = 16;              // record ring between consumers and bookkeeper
constexpr int kGrab = 4;               // units taken from the global counter at once, away from the end
constexpr int kVecPT = kVerifyStageBytes / 16 / kCT;  // 16-byte vectors per consumer thread per stage
constexpr int kWarpsB = 6;             // workers per CTA of the draw kernel
constexpr int kThreadsB = 32 * kWarpsB;
constexpr int kCtasPerSmB = 2;
constexpr int kSmemSeqs = 512;         // batches up to this size keep offsets in shared memory
constexpr int kSmemToks = 1024;        // batches up to this many positions keep their tokens there
constexpr int kPartWords = 4;          // flagged words per piece result
static_assert(kVecPT * 16 * kCT == kVerifyStageBytes, "stage split");

enum : int { kEnd = 0, kUnit = 1 };

struct Desc {
    int kind;
    int seq;         // the sequence
    int expect;      // chunks of the sequence
    int slot;        // row slot of the partial: 2 r + {0: p, 1: q}
    int chunk;
    int last;        // 1: the run of consecutive chunks of this row ends here
    int e0;          // first element of the chunk in its row
    int n;           // elements of the chunk
    int nvec;        // 16-byte vectors in shared memory
    int nsm;         // elements of the chunk in shared memory
    int skip;        // elements before e0 in the first vector
    const char* tail;  // global address of the first element not in shared memory
    float c2;        // log2(e) / T, or 0 for an argmax
};

// A run: consecutive chunks [chunk, chunk + n) of one row slot, reduced by
// one CTA in a row; its partial covers them all.
struct Rec {
    int kind, seq, expect, slot, chunk, n, arg;
    float2 wp[kCW];  // one partial per consumer warp
};

// The batch layout both kernels read: offsets and temperatures of small
// batches, proposed tokens, the valid count.
struct Tables {
    long long units;  // chunks the stream kernel reduces
    int n_valid;
    int batch_bad;
    int offs[kSmemSeqs + 1];
    float temp[kSmemSeqs];
    int tok[kSmemToks];
};

struct SmemA {
    alignas(128) unsigned char stage[kStagesV][kVerifyStageBytes];
    uint64_t full[kStagesV];
    uint64_t empty[kStagesV];
    uint64_t rec_full[kRecs];
    uint64_t rec_empty[kRecs];
    Desc desc[kStagesV];
    Rec rec[kRecs];
    Tables tb;
};

struct SmemB {
    // Each worker's two piece buffers (rows p, q).  A worker's draws come
    // after its last piece, with no copy in flight, so the piece results a
    // draw reads live in its first buffer.
    alignas(128) unsigned char buf[kWarpsB][2][2][kPieceBytes];
    uint64_t bar[kWarpsB][2];  // completion of each buffer's copies
    Tables tb;
};

// A decoded tail descriptor.
struct Tail {
    int prow, qrow, mode, qnew, tag, pos, npub, seq, dest;
    float c2, nz0, nz1;
};

template <typename Elem>
__device__ __forceinline__ float load_elem(const void* p) {
    if constexpr (sizeof(Elem) == 2)
        return __uint_as_float(static_cast<uint32_t>(*static_cast<const uint16_t*>(p)) << 16);
    else
        return *static_cast<const float*>(p);
}

__device__ __forceinline__ bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Sum of N values as a balanced tree (short dependency chains).
template <int N>
__device__ __forceinline__ float tree_sum(const float* v) {
    if constexpr (N == 1) {
        return v[0];
    } else {
        return tree_sum<N / 2>(v) + tree_sum<N - N / 2>(v + N / 2);
    }
}


// Residual weight max(0, p - q) of one id, and p itself.  nz0, nz1: log2 of
// the normalisers of p and q in the exp2 domain, so p(v) = exp2(x_v c2 - nz0).
__device__ __forceinline__ float resid_w(float xp, float xq, float c2, float nz0, float nz1, float& pv) {
    pv = soft_w(xp, c2, nz0);
    const float qv = soft_w(xq, c2, nz1);
    return fmaxf(0.0f, __fsub_rn(pv, qv));
}

// log2 by the hardware approximation (absolute error about 2^-22, subnormal
// inputs kept).
__device__ __forceinline__ float lg2_approx(float x) {
    float y;
    asm("lg2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// log2(-ln u) of a Gumbel uniform u in (0, 1): -log2(-ln u) is the Gumbel
// noise in log2 units.  Below 1/2, -ln u = -ln 2 log2 u keeps its relative
// accuracy; near u = 1 it is taken as -log1p(u - 1), u - 1 being exact there.
__device__ __forceinline__ float log2_neg_ln(float u) {
    const float nl = u < 0.5f ? -0.6931471805599453f * lg2_approx(u) : -log1pf(-(1.0f - u));
    return lg2_approx(nl);
}

// The Gumbel uniforms of ids 4b .. 4b+3 of one draw: counter (offset,
// sequence, position, 16 + purpose + 256 b), key (seed, 0), one output word
// per id; u = (top 23 bits + 1/2) 2^-23, exact in float, inside (0, 1).
__device__ __forceinline__ void gumbel_block(const VerifyArgs& a, const Tail& t, int b, float u[4]) {
    uint64_t w[4];
    philox4x64_10(a.offset, static_cast<uint64_t>(t.seq), static_cast<uint64_t>(t.pos),
                  16ull + static_cast<uint64_t>(t.tag) + 256ull * static_cast<uint64_t>(b), a.seed, 0, w);
#pragma unroll
    for (int j = 0; j < 4; ++j)
        u[j] = (static_cast<float>(static_cast<uint32_t>(w[j] >> 41)) + 0.5f) * (1.0f / 8388608.0f);
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

__device__ __forceinline__ SeqInfo seq_lookup(const VerifyArgs& a, const Tables& tb, int i) {
    return a.num_seqs <= kSmemSeqs ? seq_info_t(tb.offs, tb.temp, i, a.total)
                                   : seq_info(a.seq_offsets, a.temperature, i, a.total);
}

// Rows a valid sequence streams: p_k and q_k (T > 0), or p_1 .. p_{L+1} (T = 0).
__device__ __forceinline__ int rows_of(const SeqInfo& s) { return s.T > 0.0f ? 2 * s.len : s.len + 1; }

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

// =============================================================================
// Decision (one warp; lane k handles position k + 1)
// =============================================================================

// Publish tail `slot`: eight flagged words (two per 16-byte store).
__device__ __forceinline__ void publish_tail(const VerifyArgs& a, int slot, const uint32_t w[kTailWords]) {
    const uint32_t f = static_cast<uint32_t>(slot) + 1u;
    uint64_t* d = a.tdesc + static_cast<size_t>(slot) * kTailWords;
#pragma unroll
    for (int k = 0; k < kTailWords; k += 2) st_volatile_v2u64(d + k, flagged(f, w[k]), flagged(f, w[k + 1]));
}

// What a decision reads from its inputs alone (not from the stream kernel's
// partials): the proposed tokens, their logits, the acceptance uniforms, and
// the reservation of the sequence's queue slot.  Its loads are issued before
// the partials are staged, so that the two round trips overlap.
struct DecPrep {
    int x;       // this lane's proposed token x_{lane+1}
    float zp;    // its logit in p_{lane+1}
    float zq;    // its logit in q_{lane+1}
    float u;     // its acceptance uniform
    int tslot;   // lane 0: the queue slot of the sequence's correction or bonus draw
    int bad;     // some proposed token is outside the vocabulary
};

template <typename Elem>
__device__ __forceinline__ DecPrep decide_prep(const VerifyArgs& a, const Tables& tb, int i, int lane) {
    constexpr int E = sizeof(Elem);
    const SeqInfo s = seq_lookup(a, tb, i);
    const int L = s.len;
    const float T = s.T;
    const int r = s.start + lane;
    const bool mine = lane < L;
    DecPrep d;
    d.x = mine ? (a.total <= kSmemToks ? tb.tok[r] : __ldg(a.tokens + r)) : 0;
    d.bad = __any_sync(0xffffffffu, mine && (d.x < 0 || d.x >= a.vocab));
    // A T > 0 sequence always makes one draw after its decision: its queue
    // slot is reserved now, so that the round trip overlaps the loads below
    // (the check hook's held-back decision reserves it too, and the workers
    // that take its pieces wait for a descriptor that never comes).
    d.tslot = 0;
    if (T > 0.0f && lane == 0 && !d.bad) d.tslot = atomicAdd(&a.ctl->tail_reserve, 1);
    d.zp = 0.0f;
    d.zq = 0.0f;
    if (mine && T > 0.0f && !d.bad) {
        d.zp = load_elem<Elem>(a.p + static_cast<int64_t>(r + i) * a.ldp_bytes + static_cast<size_t>(d.x) * E);
        d.zq = load_elem<Elem>(a.q + static_cast<int64_t>(r) * a.ldq_bytes + static_cast<size_t>(d.x) * E);
    }
    d.u = (mine && T > 0.0f) ? decision_uniform(a.seed, a.offset, i, lane + 1, kTagAccept) : 0.0f;
    return d;
}

// Inlined into the worker, so that the arguments are read as kernel
// parameters (an out-of-line call would reach them through a generic pointer,
// reloaded after every store).
template <typename Elem>
__device__ __forceinline__ void decide(const VerifyArgs& a, const Tables& tb, float2* sblk, int i, const DecPrep pre,
                                       int lane) {
    // The sequence's ready word is published: every partial of it is in
    // place.
    const SeqInfo s = seq_lookup(a, tb, i);
    const int L = s.len;
    const float T = s.T;
    const float c2 = T > 0.0f ? inv_temp_log2e(T) : 0.0f;
    const int r = s.start + lane;
    const bool mine = lane < L;
    const int x = pre.x;
    if (pre.bad) {
        write_invalid(a, i, s, lane, -1);
        if (lane == 0) finalize(a);
        return;
    }
    const bool stall = i == a.stall_seq;
    int tslot = pre.tslot;
    // The sequence's partials are one contiguous block, [2 L rows][nck]: it
    // is staged in this warp's shared buffer in one round trip when it fits.
    const float2* blk = a.part + static_cast<size_t>(2 * s.start) * a.nck;
    const int nblk = 2 * L * a.nck;
    const bool staged = nblk * static_cast<int>(sizeof(float2)) <= 2 * kPieceBytes;
    if (staged)
        for (int v = lane; v < nblk / 2; v += 32) cp_async16(sblk + 2 * v, blk + 2 * v);
    const float zp = pre.zp, zq = pre.zq, u_acc = pre.u;
    if (staged) cp_async_wait_all();
    __syncwarp();
    const float2* part_of = staged ? sblk : blk;
    float ratio = 0.0f, racc = 0.0f, Mp = -INFINITY, Sp = 0.0f, Mq = -INFINITY, Sq = 0.0f;
    int amax = INT_MAX;
    if (mine) {
        const float2* pp = part_of + static_cast<size_t>(2 * lane) * a.nck;
        const float2* pq = pp + a.nck;
        auto part = [&](const float2* b, int j) -> float2 { return staged ? b[j] : __ldcg(b + j); };
        if (T > 0.0f) {
            // Two passes, so that the exponentials are independent of each
            // other: the largest mc, then the sum rescaled to it.
#pragma unroll 4
            for (int j = 0; j < a.nck; ++j) {
                Mp = fmaxf(Mp, part(pp, j).x);
                Mq = fmaxf(Mq, part(pq, j).x);
            }
            float sp4[4] = {0.0f, 0.0f, 0.0f, 0.0f}, sq4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll 4
            for (int j = 0; j < a.nck; ++j) {
                const float2 u = part(pp, j), v = part(pq, j);
                if (u.x != -INFINITY) sp4[j & 3] += u.y * ex2_approx(u.x - Mp);
                if (v.x != -INFINITY) sq4[j & 3] += v.y * ex2_approx(v.x - Mq);
            }
            Sp = tree_sum<4>(sp4);
            Sq = tree_sum<4>(sq4);
        } else {
            float M = -INFINITY;
            for (int j = 0; j < a.nck; ++j) {
                const float2 u = part(pp, j);
                merge_argmax(M, amax, u.x, __float_as_int(u.y));
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
    if (mine) acc = T > 0.0f ? u_acc < racc : ratio == 1.0f;
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
    if (T == 0.0f) {
        // Greedy: the correction is the argmax of p_j, already known; the
        // bonus is the argmax of p_{L+1}, streamed in the last position's q
        // slot.
        int tok = amax_j;
        if (na == L) {
            const float2* pb = part_of + static_cast<size_t>(2 * (L - 1) + 1) * a.nck;
            float M = -INFINITY;
            int I = INT_MAX;
            for (int g = lane; g < a.nck; g += 32) {
                const float2 v = staged ? pb[g] : __ldcg(pb + g);
                merge_argmax(M, I, v.x, __float_as_int(v.y));
            }
            warp_merge_arg(M, I);
            tok = I;
        }
        if (lane == 0) a.out_tokens[s.start + i + na] = tok;
    }
    if (stall) return;  // check hook: the reserved draw is never published, its pieces' workers wait
    // Draws left: the correction or bonus (T > 0), then one per proposal row.
    const int n_tok = T > 0.0f ? 1 : 0;
    const int n_prop = props ? L : 0;
    const int n_pub = n_tok + n_prop;
    if (n_pub == 0) {
        if (lane == 0) finalize(a);
        return;
    }
    int pbase = 0;
    if (n_prop > 0 && lane == 0) pbase = atomicAdd(&a.ctl->tail_reserve, n_prop);
    tslot = __shfl_sync(0xffffffffu, tslot, 0);
    pbase = __shfl_sync(0xffffffffu, pbase, 0);
    float nz0 = 0.0f, nz1 = 0.0f;
    if (na < L) {
        nz0 = __fadd_rn(mc0, log2f(sp0));
        nz1 = __fadd_rn(mc1, log2f(sq0));
    }
    for (int k = lane; k < n_pub; k += 32) {
        uint32_t w[kTailWords];
        int slot;
        if (k < n_tok) {
            slot = tslot;
            const int mode = na < L ? kTailRes : kTailSoft;
            const int tag = na < L ? static_cast<int>(kTagCorrect) : static_cast<int>(kTagBonus);
            w[kTwPRow] = static_cast<uint32_t>(s.start + i + na);  // p_j, or p_{L+1} when na == L
            w[kTwQRow] = static_cast<uint32_t>(s.start + na);
            w[kTwMeta] = static_cast<uint32_t>(mode | (tag << 8) | ((na + 1) << 16) | (n_pub << 24));
            w[kTwNz0] = __float_as_uint(nz0);
            w[kTwNz1] = __float_as_uint(nz1);
            w[kTwDest] = static_cast<uint32_t>(s.start + i + na);
        } else {
            const int m = k - n_tok;  // position m + 1, qnew row start + m
            slot = pbase + m;
            const int mode = T > 0.0f ? kTailSoft : kTailArg;
            w[kTwPRow] = static_cast<uint32_t>(s.start + m);
            w[kTwQRow] = 0;
            w[kTwMeta] = static_cast<uint32_t>(mode | (1 << 4) | (static_cast<int>(kTagPropose) << 8) |
                                               ((m + 1) << 16) | (n_pub << 24));
            w[kTwNz0] = 0;
            w[kTwNz1] = 0;
            w[kTwDest] = static_cast<uint32_t>(-1 - (s.start + m));
        }
        w[kTwC2] = __float_as_uint(c2);
        w[kTwSeq] = static_cast<uint32_t>(i);
        publish_tail(a, slot, w);
    }
}

// =============================================================================
// Bookkeeper warp (stream kernel): merges the eight warp partials of a unit
// and stores the unit's partial
// =============================================================================

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
// group g (8 lanes, one per consumer warp) handles record r + g.  A run's
// partial goes to its first chunk; its other chunks get a partial that holds
// nothing (max -inf; sum 0, or index INT_MAX).  Each run's chunks then count
// toward its sequence (the stores first, then the count: release); the count
// that completes a sequence publishes its ready word, on which the draw
// kernel's decision waits while the stream goes on.
__device__ void bookkeeper(const VerifyArgs& a, SmemA& sm, int lane) {
    const int g = lane >> 3, wl = lane & 7;
    for (long long r = 0;;) {
        const bool ok = __all_sync(0xffffffffu, mbar_wait_ns(&sm.rec_full[r % kRecs],
                                                             static_cast<uint32_t>(r / kRecs) & 1u, kWaitNs));
        if (!ok) {
            if (lane == 0) atomicOr(&a.ctl->err, kErrWaitTimeout);
            break;
        }
        int nb = 1;
        while (nb < 4 && mbar_test(&sm.rec_full[(r + nb) % kRecs], static_cast<uint32_t>((r + nb) / kRecs) & 1u))
            ++nb;
        const bool mine = g < nb;
        const Rec& rc = sm.rec[(r + (mine ? g : 0)) % kRecs];
        const int kind = rc.kind, rseq = rc.seq, rexpect = rc.expect, rslot = rc.slot, chunk = rc.chunk,
                  nrun = rc.n, arg = rc.arg;
        const float2 v = rc.wp[wl];
        __syncwarp();
        if (lane < nb) mbar_arrive(&sm.rec_empty[(r + lane) % kRecs]);
        // An end marker is the last record: the batch stops there.
        const unsigned end_mask = __ballot_sync(0xffffffffu, mine && wl == 0 && kind == kEnd);
        const int n_real = end_mask ? (__ffs(end_mask) - 1) / 8 : nb;
        // Both merges run on every lane (shuffles need the whole warp); each
        // group keeps the one its record asks for.
        float Mm = v.x, Sm = v.y;
        group8_merge_mc(Mm, Sm);
        float Ma = v.x;
        int Ia = __float_as_int(v.y);
        group8_merge_arg(Ma, Ia);
        if (g < n_real) {
            float2* dst = a.part + static_cast<size_t>(rslot) * a.nck + chunk;
            if (wl == 0) *dst = arg ? make_float2(Ma, __int_as_float(Ia)) : make_float2(Mm, Sm);
            const float2 none = make_float2(-INFINITY, arg ? __int_as_float(INT_MAX) : 0.0f);
            for (int j = 1 + wl; j < nrun; j += 8) dst[j] = none;
        }
        __syncwarp();
        if (g < n_real && wl == 0) {
            // The count releases this run's partials (the group's stores,
            // ordered by the warp barrier above); the count that completes
            // the sequence also acquires the other runs' and publishes the
            // ready word with a release store.
            if (atomic_add_acq_rel(a.seq_count + rseq, nrun) + nrun == rexpect)
                st_release_u64(a.dready + rseq, flagged(static_cast<uint32_t>(rseq) + 1u, 0u));
        }
        __syncwarp();
        r += nb;
        if (end_mask) break;
    }
}

// =============================================================================
// Producer thread (stream kernel): streams chunks into the stage ring
// =============================================================================

// The producer's position in the stage ring: the next stage and the phase
// of its use.
struct Ring {
    int stage = 0;
    uint32_t phase = 0;
    __device__ void advance() {
        if (++stage == kStagesV) {
            stage = 0;
            phase ^= 1u;
        }
    }
};

__device__ __forceinline__ int acquire_stage(SmemA& sm, const Ring& rg, int* err) {
    if (!mbar_wait_ns(&sm.empty[rg.stage], rg.phase ^ 1u, kWaitNs)) {
        atomicOr(err, kErrWaitTimeout);
        return -1;
    }
    return rg.stage;
}

template <typename Elem>
__device__ void producer(const VerifyArgs& a, SmemA& sm) {
    constexpr int E = sizeof(Elem);
    Ring rg;  // stages issued
    bool ok = true;
    // Each chunk is read once: its lines are the first the L2 gives up, so
    // that the stream leaves resident what the draw kernel reads next (its
    // code, the partials) instead of the rows it has finished with.
    const uint64_t stream_policy = l2_policy_evict_first();
    if (!sm.tb.batch_bad) {
        // Units in sequence order: sequence i owns [base, base + units);
        // within it, row index ri in [0, rows_of), chunk c in [0, nck).  A
        // batch of units is taken from the global counter one batch ahead of
        // its use, so a CTA that falls behind takes fewer; near the end the
        // batches shrink to single units, so that CTAs finish together.
        int i = -1;
        long long base = 0, units = 0;
        SeqInfo s{};
        float c2 = 0.0f;
        const long long fine = sm.tb.units - 2LL * kGrab * gridDim.x;  // single units from here on
        unsigned long long g = fine > 0 ? kGrab : 1;
        unsigned long long next = atomicAdd(&a.ctl->grab, g);
        unsigned long long cur = 0, cur_end = 0;
        while (ok) {
            if (cur == cur_end) {
                cur = next;
                cur_end = next + g;
                g = static_cast<long long>(next) >= fine ? 1 : kGrab;
                next = atomicAdd(&a.ctl->grab, g);
            }
            const long long U = static_cast<long long>(cur++);
            bool more = true;
            while (U >= base + units) {
                base += units;
                if (++i >= a.num_seqs) {
                    more = false;
                    break;
                }
                s = seq_lookup(a, sm.tb, i);
                units = s.ok ? static_cast<long long>(rows_of(s)) * a.nck : 0;
                c2 = s.T > 0.0f ? inv_temp_log2e(s.T) : 0.0f;
            }
            if (!more) break;
            const int u = static_cast<int>(U - base);
            const int ri = u / a.nck, c = u - ri * a.nck;
            const char* row;
            int slot;
            if (s.T > 0.0f) {  // p_k, q_k interleaved: ri = 2 (k - 1) + {0, 1}
                const int k = (ri >> 1) + 1, kind = ri & 1;
                slot = 2 * (s.start + k - 1) + kind;
                row = kind ? a.q + static_cast<int64_t>(s.start + k - 1) * a.ldq_bytes
                           : a.p + static_cast<int64_t>(s.start + i + k - 1) * a.ldp_bytes;
            } else {  // p_1 .. p_{L+1}; the final anchor uses the last position's q slot
                const int k = ri + 1;
                slot = k <= s.len ? 2 * (s.start + k - 1) : 2 * (s.start + s.len - 1) + 1;
                row = a.p + static_cast<int64_t>(s.start + i + k - 1) * a.ldp_bytes;
            }
            const int e0 = c * a.ck;
            const int nel = min(a.ck, a.vocab - e0);
            const Piece pc = make_piece<E>(row, e0, nel);
            const int stage = acquire_stage(sm, rg, &a.ctl->err);
            if (stage < 0) {
                ok = false;
                break;
            }
            Desc& d = sm.desc[stage];
            d.kind = kUnit;
            d.seq = i;
            d.expect = static_cast<int>(units);
            d.slot = slot;
            d.chunk = c;
            // The run goes on while the next unit of this CTA is the next
            // chunk of the same row.
            d.last = c == a.nck - 1 ||
                     (cur == cur_end && (next != cur_end || static_cast<long long>(next) >= sm.tb.units));
            d.e0 = e0;
            d.n = nel;
            d.nvec = pc.bytes >> 4;
            d.nsm = pc.nsm;
            d.skip = pc.skip;
            d.tail = pc.tail;
            d.c2 = c2;
            if (pc.bytes > 0) {
                mbar_arrive_expect_tx(&sm.full[stage], static_cast<uint32_t>(pc.bytes));
                bulk_copy_g2s_hint(sm.stage[stage], reinterpret_cast<const void*>(pc.lo),
                                   static_cast<uint32_t>(pc.bytes), &sm.full[stage], stream_policy);
            } else {
                mbar_arrive(&sm.full[stage]);
            }
            rg.advance();
        }
    }
    const int stage = acquire_stage(sm, rg, &a.ctl->err);
    if (stage >= 0) {
        sm.desc[stage].kind = kEnd;
        mbar_arrive(&sm.full[stage]);
    }
}

// =============================================================================
// Consumer warps
// =============================================================================

// Hand this warp's partial of a run to the bookkeeper.
__device__ __forceinline__ void push_record(const VerifyArgs& a, SmemA& sm, long long& nrec, int warp, int lane,
                                            float2 part, int kind, int seq, int expect, int slot, int chunk, int n,
                                            int arg) {
    const int rs = static_cast<int>(nrec % kRecs);
    const uint32_t parity = (static_cast<uint32_t>(nrec / kRecs) & 1u) ^ 1u;
    ++nrec;
    if (lane == 0) {
        if (!mbar_wait_ns(&sm.rec_empty[rs], parity, kDrainWaitNs)) atomicOr(&a.ctl->err, kErrWaitTimeout);
        Rec& rc = sm.rec[rs];
        rc.wp[warp] = part;
        if (warp == 0) {
            rc.kind = kind;
            rc.seq = seq;
            rc.expect = expect;
            rc.slot = slot;
            rc.chunk = chunk;
            rc.n = n;
            rc.arg = arg;
        }
        mbar_arrive(&sm.rec_full[rs]);
    }
    __syncwarp();
}

// Largest of 2 kN bf16 (or kN fp32) values, as a tree.
template <bool kBf16, int kN>
__device__ __forceinline__ float tree_max(const uint32_t* w) {
    if constexpr (kBf16) {
        uint32_t m[kN];
#pragma unroll
        for (int j = 0; j < kN; ++j) m[j] = w[j];
#pragma unroll
        for (int h = kN / 2; h > 0; h >>= 1)
#pragma unroll
            for (int j = 0; j < h; ++j) m[j] = hmax2_bf16(m[j], m[j + h]);
        return fmaxf(bf16lo(m[0]), bf16hi(m[0]));
    } else {
        float m[kN];
#pragma unroll
        for (int j = 0; j < kN; ++j) m[j] = __uint_as_float(w[j]);
#pragma unroll
        for (int h = kN / 2; h > 0; h >>= 1)
#pragma unroll
            for (int j = 0; j < h; ++j) m[j] = fmaxf(m[j], m[j + h]);
        return m[0];
    }
}

// The open run of a consumer thread: softmax partial (RM = largest x c2
// so far, RS = sum of exp2(x c2 - RM)), or argmax partial (RM, RI: the
// first position of the largest value).
struct Run {
    float RM;
    float RS;
    int RI;
};

// Sum over this thread's share of a chunk of exp2(x c2 - ref), in packed
// pairs: one fused multiply-add and one addition per two elements.
template <bool kBf16>
__device__ __forceinline__ float chunk_sum(const uint32_t* w, float tv, float c2, float ref) {
    const float2 C2 = make_float2(c2, c2), NMC = make_float2(-ref, -ref);
    float2 acc[4] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f),
                     make_float2(0.0f, 0.0f)};
#pragma unroll
    for (int j = 0; j < kVecPT * 4; ++j) {
        float2 x;
        if constexpr (kBf16) {
            x = make_float2(bf16lo(w[j]), bf16hi(w[j]));
        } else {
            if (j & 1) continue;
            x = make_float2(__uint_as_float(w[j]), __uint_as_float(w[j + 1]));
        }
        const float2 y = __ffma2_rn(x, C2, NMC);
        acc[j & 3] = __fadd2_rn(acc[j & 3], make_float2(ex2_approx(y.x), ex2_approx(y.y)));
    }
    if (tv != -INFINITY) acc[1].x += soft_w(tv, c2, ref);
    const float2 t = __fadd2_rn(__fadd2_rn(acc[0], acc[1]), __fadd2_rn(acc[2], acc[3]));
    return t.x + t.y;
}

// One stage: this thread's share of the chunk (kVecPT 16-byte vectors, and
// at most one element after the last whole vector) folded into its run.
template <typename Elem>
__device__ __forceinline__ void unit_stage(SmemA& sm, int stage, const Desc& d, int tid, int lane, Run& r) {
    constexpr bool kBf16 = sizeof(Elem) == 2;
    constexpr uint32_t kNeg = kBf16 ? 0xff80ff80u : 0xff800000u;  // -inf pattern
    uint32_t w[kVecPT * 4];
    const uint4* sv = reinterpret_cast<const uint4*>(sm.stage[stage]);
    if (d.nvec == kVecPT * kCT) {  // a full stage
#pragma unroll
        for (int k = 0; k < kVecPT; ++k) {
            const uint4 v = sv[tid + k * kCT];
            w[4 * k] = v.x;
            w[4 * k + 1] = v.y;
            w[4 * k + 2] = v.z;
            w[4 * k + 3] = v.w;
        }
    } else {
#pragma unroll
        for (int k = 0; k < kVecPT; ++k) {
            const int vi = tid + k * kCT;
            const uint4 v = vi < d.nvec ? sv[vi] : make_uint4(kNeg, kNeg, kNeg, kNeg);
            w[4 * k] = v.x;
            w[4 * k + 1] = v.y;
            w[4 * k + 2] = v.z;
            w[4 * k + 3] = v.w;
        }
    }
    if (d.skip != 0 && tid == 0) {  // elements before the chunk in the first vector
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if constexpr (kBf16) {
                if (2 * j < d.skip) w[j] = (w[j] & 0xffff0000u) | 0xff80u;
                if (2 * j + 1 < d.skip) w[j] = (w[j] & 0x0000ffffu) | 0xff800000u;
            } else {
                if (j < d.skip) w[j] = kNeg;
            }
        }
    }
    const int ntail = d.n - d.nsm;
    float tv = -INFINITY;
    if (tid < ntail) tv = load_elem<Elem>(d.tail + static_cast<size_t>(tid) * sizeof(Elem));
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.empty[stage]);

    const float c2 = d.c2;
    if (c2 > 0.0f) {
        // The chunk is summed against the run's largest value so far; the
        // first chunk of a run takes the largest of its first four words.
        // A sum past 2^64 (a value far above the reference) is summed again
        // against the chunk's own largest value.
        float ref = r.RM;
        if (ref == -INFINITY) ref = fmaxf(tree_max<kBf16, 4>(w), tv) * c2;
        float sc = ref == -INFINITY ? INFINITY : chunk_sum<kBf16>(w, tv, c2, ref);
        if (!(sc <= 18446744073709551616.0f)) {
            ref = fmaxf(tree_max<kBf16, kVecPT * 4>(w), tv) * c2;
            sc = ref == -INFINITY ? 0.0f : chunk_sum<kBf16>(w, tv, c2, ref);
        }
        if (ref > r.RM) {  // a new reference: rescale the run's sum
            r.RS = r.RS * ex2_approx(r.RM - ref) + sc;
            r.RM = ref;
        } else {
            r.RS += sc;
        }
        return;
    }
    const float cm = fmaxf(tree_max<kBf16, kVecPT * 4>(w), tv);
    if (cm > r.RM) {
        // First position of the maximum in this thread's (ascending)
        // elements; a later chunk of the run takes over only if larger.
        constexpr int kPer = kBf16 ? 8 : 4;
        int idx = d.nsm + tid;  // the element after the vectors, unless a vector holds the maximum
#pragma unroll
        for (int k = kVecPT - 1; k >= 0; --k) {
#pragma unroll
            for (int j = 3; j >= 0; --j) {
                const uint32_t x = w[4 * k + j];
                const int base = (tid + k * kCT) * kPer - d.skip;
                if constexpr (kBf16) {
                    if (bf16hi(x) == cm) idx = base + 2 * j + 1;
                    if (bf16lo(x) == cm) idx = base + 2 * j;
                } else {
                    if (__uint_as_float(x) == cm) idx = base + j;
                }
            }
        }
        r.RM = cm;
        r.RI = d.e0 + idx;
    }
}

template <typename Elem>
__device__ void consumer(const VerifyArgs& a, SmemA& sm, int tid, int warp, int lane) {
    long long nrec = 0;
    Run r{-INFINITY, 0.0f, INT_MAX};
    int run_chunk = -1;  // first chunk of the open run
    int stage = 0;
    uint32_t parity = 0;
    for (;; stage = stage + 1 == kStagesV ? (parity ^= 1u, 0) : stage + 1) {
        if (!__all_sync(0xffffffffu, mbar_wait_ns(&sm.full[stage], parity, kDrainWaitNs + kWaitNs))) {
            if (lane == 0) atomicOr(&a.ctl->err, kErrWaitTimeout);
            break;
        }
        const Desc d = sm.desc[stage];
        if (d.kind == kEnd) break;
        if (run_chunk < 0) run_chunk = d.chunk;
        unit_stage<Elem>(sm, stage, d, tid, lane, r);
        if (d.last) {
            const bool arg = d.c2 == 0.0f;
            float M = r.RM, S = r.RS;
            int I = r.RI;
            float2 part;
            if (arg) {
                warp_merge_arg(M, I);
                part = make_float2(M, __int_as_float(I));
            } else {
                warp_merge_mc(M, S);
                part = make_float2(M, S);
            }
            push_record(a, sm, nrec, warp, lane, part, kUnit, d.seq, d.expect, d.slot, run_chunk,
                        d.chunk - run_chunk + 1, arg);
            r = Run{-INFINITY, 0.0f, INT_MAX};
            run_chunk = -1;
        }
    }
    // Tell the bookkeeper there is no more work (a record of kind kEnd).
    push_record(a, sm, nrec, warp, lane, make_float2(0.0f, 0.0f), kEnd, 0, 0, 0, 0, 0, 0);
}

// =============================================================================
// Workers: tail pieces and draws
// =============================================================================

__device__ __forceinline__ Tail decode_tail(uint64_t w, int lane) {
    const uint32_t x = static_cast<uint32_t>(w);
    Tail t;
    t.prow = static_cast<int>(__shfl_sync(0xffffffffu, x, kTwPRow));
    t.qrow = static_cast<int>(__shfl_sync(0xffffffffu, x, kTwQRow));
    const uint32_t meta = __shfl_sync(0xffffffffu, x, kTwMeta);
    t.mode = static_cast<int>(meta & 15u);
    t.qnew = static_cast<int>((meta >> 4) & 1u);
    t.tag = static_cast<int>((meta >> 8) & 255u);
    t.pos = static_cast<int>((meta >> 16) & 255u);
    t.npub = static_cast<int>(meta >> 24);
    t.c2 = __uint_as_float(__shfl_sync(0xffffffffu, x, kTwC2));
    t.nz0 = __uint_as_float(__shfl_sync(0xffffffffu, x, kTwNz0));
    t.nz1 = __uint_as_float(__shfl_sync(0xffffffffu, x, kTwNz1));
    t.seq = static_cast<int>(__shfl_sync(0xffffffffu, x, kTwSeq));
    t.dest = static_cast<int>(__shfl_sync(0xffffffffu, x, kTwDest));
    return t;
}

template <typename Elem>
__device__ __forceinline__ const char* tail_prow(const VerifyArgs& a, const Tail& t) {
    return t.qnew ? a.qnew + static_cast<int64_t>(t.prow) * a.ldqnew_bytes
                  : a.p + static_cast<int64_t>(t.prow) * a.ldp_bytes;
}

// ---- tail pieces ----------------------------------------------------------------
// A piece is ids [k ps, k ps + ps) of a tail's row or row pair (kPieceBytes
// of each row).  A worker double-buffers its pieces: while it reduces one,
// the bulk copies of the next are in flight.  Its lanes read a staged piece
// as 16-byte vectors in lane order, so that step j (vectors 32 j .. 32 j +
// 31, 512 bytes of ids) is block j of the piece: the unit a draw walks after
// choosing the piece.

constexpr int kBlk = kPieceBlocks;        // blocks per piece
constexpr int kRecWords = kPieceRecWords;  // flagged words per piece record: result, then block weights
static_assert(kRecWords == kPartWords + kBlk, "record layout");
static_assert(kBlk % 4 == 0, "blocks are reduced four at a time");

// A piece a worker holds: its ticket and tail, where its ids are, and how
// much of each row its buffer stages.
struct Held {
    unsigned long long ticket;
    int state;          // kHeldNone, kHeldWait (descriptor not yet seen), kHeldLoad (copies issued)
    int slot, k;
    Tail t;
    const char* gp;     // first id of the piece in the drawn row
    const char* gq;     // the same in q_j (residual)
    int len;            // ids in the piece
    int nbytes;         // staged bytes of each row: whole 16-byte vectors, 0 when the rows are read in place
};
enum : int { kHeldNone = 0, kHeldWait = 1, kHeldLoad = 2 };

// Ids v VEC .. v VEC + VEC - 1 of one row of a piece (-inf past len) from
// global memory (a draw's block).
template <typename Elem>
__device__ __forceinline__ void piece_vec_global(const char* g, int len, int v, float x[16 / sizeof(Elem)]) {
    constexpr int E = sizeof(Elem), VEC = 16 / E;
    if (aligned16(g) && (v + 1) * VEC <= len) {
        const uint4 u = __ldcg(reinterpret_cast<const uint4*>(g) + v);
#pragma unroll
        for (int jv = 0; jv < VEC; ++jv) x[jv] = vec_elem<E>(u, jv);
    } else {
#pragma unroll
        for (int jv = 0; jv < VEC; ++jv) {
            const int e = v * VEC + jv;
            x[jv] = e < len ? load_elem<Elem>(g + static_cast<size_t>(e) * E) : -INFINITY;
        }
    }
}

// The same from a staged buffer row (every vector of it is there: copied,
// or filled by stage_rows).
template <typename Elem>
__device__ __forceinline__ void piece_vec(const unsigned char* st, int v, float x[16 / sizeof(Elem)]) {
    constexpr int E = sizeof(Elem), VEC = 16 / E;
    const uint4 u = *reinterpret_cast<const uint4*>(st + 16 * v);
#pragma unroll
    for (int jv = 0; jv < VEC; ++jv) x[jv] = vec_elem<E>(u, jv);
}

// Block sums of four blocks: lane l holds v[i], its share of block i; every
// lane returns the warp's sum for block (l >> 3) & 3 (a reduce-scatter: each
// of the first two exchanges halves the blocks a lane keeps).
__device__ __forceinline__ float block_sums4(const float (&v)[4], int lane) {
    const bool b4 = lane & 16, b3 = lane & 8;
    float w2[2];
#pragma unroll
    for (int i = 0; i < 2; ++i)
        w2[i] = (b4 ? v[i + 2] : v[i]) + __shfl_xor_sync(0xffffffffu, b4 ? v[i] : v[i + 2], 16);
    float w1 = (b3 ? w2[1] : w2[0]) + __shfl_xor_sync(0xffffffffu, b3 ? w2[0] : w2[1], 8);
    w1 += __shfl_xor_sync(0xffffffffu, w1, 4);
    w1 += __shfl_xor_sync(0xffffffffu, w1, 2);
    w1 += __shfl_xor_sync(0xffffffffu, w1, 1);
    return w1;
}

// Stage a piece's rows in buffer b: bulk copies of the whole 16-byte vectors
// (completing on bar[b]) while the lanes fill the rest of each buffer row,
// the last ids of the row from global memory and -inf past them (rows whose
// piece does not start on a 16-byte boundary are filled whole), so that a
// reduction reads every vector from shared memory.
template <typename Elem>
__device__ __noinline__ void fill_rows(SmemB& sm, int wi, int b, const char* gp, const char* gq, int len, int nbytes,
                                      bool two, int lane) {
    constexpr int E = sizeof(Elem), VEC = 16 / E;
    using Raw = typename std::conditional<E == 2, uint16_t, uint32_t>::type;
    constexpr Raw kNegInf = E == 2 ? static_cast<Raw>(0xff80u) : static_cast<Raw>(0xff800000u);
    for (int r = 0; r < (two ? 2 : 1); ++r) {
        const Raw* g = reinterpret_cast<const Raw*>(r ? gq : gp);
        unsigned char* row = sm.buf[wi][b][r];
        for (int off = nbytes + 16 * lane; off < kPieceBytes; off += 512) {
            Raw v[VEC];
#pragma unroll
            for (int jv = 0; jv < VEC; ++jv) {
                const int e = off / E + jv;
                v[jv] = e < len ? g[e] : kNegInf;
            }
            *reinterpret_cast<uint4*>(row + off) = *reinterpret_cast<const uint4*>(v);
        }
    }
}

template <typename Elem>
__device__ __forceinline__ void stage_rows(SmemB& sm, int wi, int b, Held& h, bool two, int lane) {
    constexpr int E = sizeof(Elem);
    const bool ok = aligned16(h.gp) && (!two || aligned16(h.gq));
    h.nbytes = ok ? ((h.len * E) & ~15) : 0;
    __syncwarp();
    if (h.nbytes < kPieceBytes) fill_rows<Elem>(sm, wi, b, h.gp, h.gq, h.len, h.nbytes, two, lane);
    if (lane == 0) {
        uint64_t* bar = &sm.bar[wi][b];
        if (h.nbytes > 0) {
            fence_proxy_async();  // this buffer's earlier reads come before the copy's writes
            mbar_arrive_expect_tx(bar, static_cast<uint32_t>(h.nbytes * (two ? 2 : 1)));
            bulk_copy_g2s(sm.buf[wi][b][0], h.gp, static_cast<uint32_t>(h.nbytes), bar);
            if (two) bulk_copy_g2s(sm.buf[wi][b][1], h.gq, static_cast<uint32_t>(h.nbytes), bar);
        } else {
            mbar_arrive(bar);
        }
    }
    __syncwarp();  // the filled vectors are visible to every lane
}

// Look for the descriptor of a held ticket; once it is there, issue the
// piece's copies.  A ticket past the last tail (every decision made, its
// slot beyond the reserved ones) is dropped.
template <typename Elem>
__device__ __forceinline__ void try_start(const VerifyArgs& a, SmemB& sm, int wi, int b, Held& h, int n_valid,
                                          int lane) {
    constexpr int E = sizeof(Elem);
    uint64_t w = 0;
    if (lane < kTailWords) w = ld_volatile_u64(a.tdesc + static_cast<size_t>(h.slot) * kTailWords + lane);
    const bool ready = __all_sync(0xffffffffu, lane >= kTailWords ||
                                                   static_cast<uint32_t>(w >> 32) == static_cast<uint32_t>(h.slot) + 1u);
    if (!ready) {
        int gone = 0;
        if (lane == 0 && ld_acquire(&a.ctl->ddone) >= n_valid) gone = h.slot >= ld_volatile(&a.ctl->tail_reserve);
        if (__shfl_sync(0xffffffffu, gone, 0)) h.state = kHeldNone;
        return;
    }
    h.t = decode_tail(w, lane);
    const int e0 = h.k * a.ps;
    h.len = min(a.ps, a.vocab - e0);
    h.gp = tail_prow<Elem>(a, h.t) + static_cast<size_t>(e0) * E;
    h.gq = a.q + static_cast<int64_t>(h.t.qrow) * a.ldq_bytes + static_cast<size_t>(e0) * E;
    stage_rows<Elem>(sm, wi, b, h, h.t.mode == kTailRes, lane);
    h.state = kHeldLoad;
}

// A claimed tail-piece ticket into h.
__device__ __forceinline__ void take_ticket(const VerifyArgs& a, Held& h, unsigned long long ticket,
                                            unsigned long long cap) {
    h.ticket = ticket;
    if (ticket >= cap) {
        h.state = kHeldNone;
        return;
    }
    h.slot = static_cast<int>(ticket / static_cast<unsigned long long>(a.np));
    h.k = static_cast<int>(ticket % static_cast<unsigned long long>(a.np));
    h.state = kHeldWait;
}

// Claim the next tail-piece ticket into h.
__device__ __forceinline__ void claim_piece(const VerifyArgs& a, Held& h, unsigned long long cap, int lane) {
    unsigned long long raw = 0;
    if (lane == 0) raw = atomicAdd(&a.ctl->claim, 1ull);
    take_ticket(a, h, __shfl_sync(0xffffffffu, raw, 0), cap);
}

// Reduce one staged piece and publish its record: the result as four
// flagged words,
//   inverse CDF, residual:  (sum of max(0, p - q), sum of p)
//   inverse CDF, softmax:   (mc, sum exp2(x c2 - mc)), mc = the piece's largest logit times c2
//   argmax (T = 0):         (max, lowest id)
//   Gumbel-max:             (best score, its id, best score of p alone, its id)
// (a Gumbel score is log2 w_v - log2(-ln u_v); the last pair is the fallback
// for a residual that rounds to zero everywhere), then, for the inverse CDF,
// the kBlk block weights in the piece's own scale.  Returns, on lane 0, the
// tail's count of finished pieces before this one (np - 1: this piece
// completes the tail).
template <typename Elem, bool kGum>
__device__ __forceinline__ int reduce_piece(const VerifyArgs& a, const unsigned char* sp, const unsigned char* sq,
                                             const Held h, int lane) {
    constexpr int VEC = 16 / sizeof(Elem);
    const Tail t = h.t;
    // Everything the loops read, in registers.
    const float c2 = t.c2, nz0 = t.nz0, nz1 = t.nz1;
    const int e0 = h.k * a.ps;
    const int n = h.len;
    const bool res = t.mode == kTailRes;
    const bool gum = kGum && t.mode != kTailArg;
    const uint32_t f = static_cast<uint32_t>(h.slot) + 1u;
    uint64_t* rec = a.tpart + (static_cast<size_t>(h.slot) * a.np + h.k) * kRecWords;
    uint32_t out[kPartWords] = {0, 0, 0, 0};
    if (gum || t.mode == kTailArg) {
        float best = -INFINITY, best_p = -INFINITY;
        int bid = INT_MAX, bid_p = INT_MAX;
        for (int j = 0; j < kBlk; ++j) {
            const int v = 32 * j + lane;
            const int e = v * VEC;
            if (e >= n) break;
            float xp[VEC], xq[VEC];
            piece_vec<Elem>(sp, v, xp);
            if (res) piece_vec<Elem>(sq, v, xq);
            if (gum) {
                // One Philox block (four ids) at a time keeps the live
                // registers of the uniforms and logarithms few.
#pragma unroll 1
                for (int bb = 0; bb < VEC; bb += 4) {
                    float u[4];
                    gumbel_block(a, t, (e0 + e + bb) >> 2, u);
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        const int jv = bb + jj;
                        const int id = e0 + e + jv;
                        const float g = log2_neg_ln(u[jj]);
                        float lw, lpw = -INFINITY;
                        if (res) {
                            float pv;
                            const float w = resid_w(xp[jv], xq[jv], c2, nz0, nz1, pv);
                            lw = w > 0.0f ? lg2_approx(w) : -INFINITY;
                            lpw = pv > 0.0f ? lg2_approx(pv) : -INFINITY;
                        } else {
                            lw = xp[jv] * c2;
                        }
                        const float sc = lw - g, scp = lpw - g;
                        if (lw != -INFINITY && sc > best) {
                            best = sc;
                            bid = id;
                        }
                        if (lpw != -INFINITY && scp > best_p) {
                            best_p = scp;
                            bid_p = id;
                        }
                    }
                }
            } else {  // argmax: the first maximum of this lane's ids is kept
#pragma unroll
                for (int jv = 0; jv < VEC; ++jv)
                    if (xp[jv] > best) {
                        best = xp[jv];
                        bid = e0 + e + jv;
                    }
            }
        }
        // Largest score, lowest id among equals.
        const float W = warp_max(best);
        const int I = warp_min_int(best == W ? bid : INT_MAX);
        out[0] = __float_as_uint(W);
        out[1] = static_cast<uint32_t>(I);
        if (gum && res) {
            const float Wp = warp_max(best_p);
            const int Ip = warp_min_int(best_p == Wp ? bid_p : INT_MAX);
            out[2] = __float_as_uint(Wp);
            out[3] = static_cast<uint32_t>(Ip);
        }
    } else {
        // Inverse CDF: each block's weight, stored as soon as its group of
        // four is reduced, and the piece's sums.
        float mc = 0.0f;
        if (!res) {  // the softmax reference: the piece's largest logit times c2
            float m = -INFINITY;
#pragma unroll 4
            for (int j = 0; j < kBlk; ++j) {
                float xp[VEC];
                piece_vec<Elem>(sp, 32 * j + lane, xp);
#pragma unroll
                for (int jv = 0; jv < VEC; ++jv) m = fmaxf(m, xp[jv]);
            }
            m = warp_max(m);
            mc = m == -INFINITY ? -INFINITY : m * c2;
        }
        const bool any = res || mc != -INFINITY;
        float tot = 0.0f, bp = 0.0f;
#pragma unroll 1
        for (int g = 0; g < kBlk / 4; ++g) {
            float v[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            if (any) {
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const int vi = 32 * (4 * g + jj) + lane;
                    float xp[VEC], w[VEC];
                    piece_vec<Elem>(sp, vi, xp);
                    if (res) {
                        float xq[VEC], pv[VEC];
                        piece_vec<Elem>(sq, vi, xq);
#pragma unroll
                        for (int jv = 0; jv < VEC; ++jv) w[jv] = resid_w(xp[jv], xq[jv], c2, nz0, nz1, pv[jv]);
                        bp += tree_sum<VEC>(pv);
                    } else {
#pragma unroll
                        for (int jv = 0; jv < VEC; ++jv) w[jv] = soft_w(xp[jv], c2, mc);
                    }
                    v[jj] = tree_sum<VEC>(w);
                }
            }
            const float sg = block_sums4(v, lane);
            if ((lane & 7) == 0) {
                st_volatile_u64(rec + kPartWords + 4 * g + (lane >> 3), flagged(f, __float_as_uint(sg)));
                tot += sg;
            }
        }
        // The piece's total is the sum of its block weights, as a draw sees them.
        tot = warp_sum(tot);
        if (res) {
            out[0] = __float_as_uint(tot);
            out[1] = __float_as_uint(warp_sum(bp));
        } else {
            out[0] = __float_as_uint(mc);
            out[1] = __float_as_uint(mc == -INFINITY ? 0.0f : tot);
        }
    }
    if (lane < kPartWords) st_volatile_u64(rec + lane, flagged(f, out[lane]));
    // The words carry their flags, so the count needs no ordering.
    int cnt = 0;
    if (lane == 0) cnt = atomicAdd(a.tcount + h.slot, 1);
    return cnt;
}

// The weight of one id in a draw, from its p (and q) logit: the softmax
// weight exp2(x c2 - mc) (soft), the residual max(0, p - q), or p itself
// (a residual that rounded to zero everywhere).  Passed by value.
struct DrawW {
    int kind;  // 0 soft, 1 residual, 2 p of the residual's row
    float c2, mc, nz0, nz1;
    __device__ __forceinline__ float operator()(float xp, float xq) const {
        if (kind == 0) return soft_w(xp, c2, mc);
        float pv;
        const float rw = resid_w(xp, xq, c2, nz0, nz1, pv);
        return kind == 1 ? rw : pv;
    }
};

// The weight of piece kp of a draw, from its result (soft: (mc, s) rescaled
// to the largest mc; residual: sum of max(0, p - q), or of p).
struct PieceW {
    const float4* pr;
    int kind;  // as DrawW
    float mc;
    __device__ __forceinline__ float operator()(int kp) const {
        const float4 v = pr[kp];
        if (kind == 0) return v.x == -INFINITY ? 0.0f : v.y * ex2_approx(v.x - mc);
        return kind == 1 ? v.x : v.y;
    }
};

// Inverse-CDF position of `target` in the running sum of n weights w(0 ..
// n-1) spread over the warp (lane l holds ids [l q, l q + q)): the first id
// whose running sum exceeds the target, else the last id of positive weight
// (rounding), else 0.  `local` receives the target minus the sum before the
// chosen lane's block.
template <typename F>
__device__ __forceinline__ int warp_icdf(int n, int q, float target, const F& w, int lane, float* local = nullptr) {
    const int b = lane * q;
    const int cnt = max(0, min(q, n - b));
    float own = 0.0f;
    int lp = -1;
    for (int e = 0; e < cnt; ++e) {
        const float x = w(b + e);
        own += x;
        if (x > 0.0f) lp = b + e;
    }
    float incl = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    const unsigned hit = __ballot_sync(0xffffffffu, cnt > 0 && incl > target);
    int found = -1;
    if (hit) {
        const int owner = __ffs(hit) - 1;
        const float before = __shfl_sync(0xffffffffu, incl - own, owner);
        // The owner's block, one id per lane at a time, in order.
        const int ob = owner * q;
        const int ocnt = max(0, min(q, n - ob));
        float cum = before;
        for (int e0 = 0; e0 < ocnt && found < 0; e0 += 32) {
            const int e = e0 + lane;
            const float x = e < ocnt ? w(ob + e) : 0.0f;
            float c = x;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, c, o);
                if (lane >= o) c += y;
            }
            const unsigned h = __ballot_sync(0xffffffffu, e < ocnt && cum + c > target);
            if (h) {
                const int hl = __ffs(h) - 1;
                found = ob + e0 + hl;
                // The target measured from the start of the chosen element.
                if (local) *local = target - (cum + __shfl_sync(0xffffffffu, c - x, hl));
            }
            cum += __shfl_sync(0xffffffffu, c, 31);
        }
        if (found < 0) {  // rounding inside the block: its last element of positive weight
            found = __shfl_sync(0xffffffffu, lp, owner);
            if (local) *local = INFINITY;
        }
    }
    if (found < 0) {
        const int last = warp_max_int(lp);
        found = last >= 0 ? last : 0;
        if (local) *local = INFINITY;
    }
    return found;
}

// The draw of a queued tail: reads every piece result (all counted, their
// flagged words land moments later at most), draws, writes the token, and
// clears the tail's words and count for the next call.  False if a wait ran
// out.  Inlined for the same reason as decide.
template <typename Elem, bool kGum>
__device__ __forceinline__ bool select_draw(const VerifyArgs& a, SmemB& sm, int wi, const Held hd, int lane) {
    constexpr int VEC = 16 / sizeof(Elem);
    const Tail& t = hd.t;
    const int slot = hd.slot;
    const int np = a.np;
    float4* pr = reinterpret_cast<float4*>(sm.buf[wi][0][0]);  // the buffers are idle during draws
    const uint32_t f = static_cast<uint32_t>(slot) + 1u;
    const uint64_t* src = a.tpart + static_cast<size_t>(slot) * np * kRecWords;
    const bool gum = kGum && t.mode != kTailArg;
    // The draw's uniform, while the results are on their way.
    const float rnd = (gum || t.mode == kTailArg) ? 0.0f : decision_uniform(a.seed, a.offset, t.seq, t.pos, t.tag);
    // Wait for every piece: each lane polls pieces lane, lane + 32, ...
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        bool mine = true;
        for (int kp = lane; kp < np; kp += 32) {
            uint64_t w0, w1, w2, w3;
            ld_volatile_v2u64(src + static_cast<size_t>(kp) * kRecWords, w0, w1);
            ld_volatile_v2u64(src + static_cast<size_t>(kp) * kRecWords + 2, w2, w3);
            mine = mine && (w0 >> 32) == f && (w1 >> 32) == f && (w2 >> 32) == f && (w3 >> 32) == f;
            pr[kp] = make_float4(__uint_as_float(static_cast<uint32_t>(w0)), __uint_as_float(static_cast<uint32_t>(w1)),
                                 __uint_as_float(static_cast<uint32_t>(w2)), __uint_as_float(static_cast<uint32_t>(w3)));
        }
        if (__all_sync(0xffffffffu, mine)) break;
        if (global_timer_ns() - t0 > a.wait_ns) {
            if (lane == 0) atomicOr(&a.ctl->err, kErrWaitTimeout);
            return false;
        }
        __nanosleep(64);
    }
    __syncwarp();
    int token;
    if (gum || t.mode == kTailArg) {
        // Largest (score, lowest id) over the pieces; a Gumbel residual that
        // rounded to zero everywhere draws from p_j (its second pair).
        float M = -INFINITY, Mp = -INFINITY;
        int I = INT_MAX, Ip = INT_MAX;
        for (int kp = lane; kp < np; kp += 32) {
            merge_argmax(M, I, pr[kp].x, __float_as_int(pr[kp].y));
            merge_argmax(Mp, Ip, pr[kp].z, __float_as_int(pr[kp].w));
        }
        warp_merge_arg(M, I);
        if (gum && t.mode == kTailRes && I == INT_MAX) {
            warp_merge_arg(Mp, Ip);
            I = Ip;
        }
        token = I == INT_MAX ? 0 : I;
    } else {
        // Inverse CDF: piece weights in one scale, the target u * total, its
        // piece, its block, then its id, every sum in vocabulary order.
        const bool soft = t.mode == kTailSoft;
        float MC = -INFINITY, W = 0.0f;
        for (int kp = lane; kp < np; kp += 32) {
            MC = fmaxf(MC, pr[kp].x);
            W += pr[kp].x;
        }
        bool fallback = false;
        if (soft) MC = warp_max(MC);
        else fallback = !(warp_sum(W) > 0.0f);  // residual rounded to zero: draw from p_j
        const int kind = soft ? 0 : (fallback ? 2 : 1);
        const PieceW piece_w{pr, kind, MC};
        float total = 0.0f;
        for (int kp = lane; kp < np; kp += 32) total += piece_w(kp);
        total = warp_sum(total);
        float tloc = INFINITY;
        const int chosen = warp_icdf(np, (np + 31) / 32, rnd * total, piece_w, lane, &tloc);
        Held h = hd;
        const int lo = chosen * a.ps;
        h.k = chosen;
        h.len = min(a.ps, a.vocab - lo);
        h.gp = tail_prow<Elem>(a, t) + static_cast<size_t>(lo) * sizeof(Elem);
        h.gq = a.q + static_cast<int64_t>(t.qrow) * a.ldq_bytes + static_cast<size_t>(lo) * sizeof(Elem);
        h.nbytes = 0;
        const float mc_k = soft ? pr[chosen].x : 0.0f;
        const DrawW id_w{kind, t.c2, soft ? mc_k : MC, t.nz0, t.nz1};
        float bw = 0.0f;  // lane j < kBlk: the weight of block j of the chosen piece
        if (kind == 2) {
            // A residual that rounded to zero everywhere draws from p_j: no
            // block weights of p were kept, so its blocks are summed here
            // from the row (a path that rounding alone can reach).
#pragma unroll 1
            for (int g = 0; g < kBlk / 4; ++g) {
                float v[4];
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    float xp[VEC], w[VEC];
                    piece_vec_global<Elem>(h.gp, h.len, 32 * (4 * g + jj) + lane, xp);
#pragma unroll
                    for (int jv = 0; jv < VEC; ++jv) w[jv] = id_w(xp[jv], 0.0f);
                    v[jj] = tree_sum<VEC>(w);
                }
                // Lane l < kBlk keeps block l = 4 g + (l & 3), reduced on lane (l & 3) * 8.
                const float sg = __shfl_sync(0xffffffffu, block_sums4(v, lane), (lane & 3) << 3);
                if ((lane >> 2) == g) bw = sg;
            }
            if (lane >= kBlk) bw = 0.0f;
        } else {
            // The chosen piece's block weights, published with its result.
            const uint64_t* bsrc = src + static_cast<size_t>(chosen) * kRecWords + kPartWords;
            for (;;) {
                uint64_t w = 0;
                if (lane < kBlk) w = ld_volatile_u64(bsrc + lane);
                if (__all_sync(0xffffffffu, lane >= kBlk || (w >> 32) == f)) {
                    bw = lane < kBlk ? __uint_as_float(static_cast<uint32_t>(w)) : 0.0f;
                    break;
                }
                if (global_timer_ns() - t0 > a.wait_ns) {
                    if (lane == 0) atomicOr(&a.ctl->err, kErrWaitTimeout);
                    return false;
                }
            }
        }
        // The block: the first whose running weight passes the target, in
        // the piece's own scale.
        const float tpiece = soft ? tloc * ex2_approx(MC - mc_k) : tloc;
        float incl = bw;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        const unsigned hit = __ballot_sync(0xffffffffu, lane < kBlk && incl > tpiece);
        int bb;
        float tb;
        if (hit) {
            bb = __ffs(hit) - 1;
            tb = tpiece - __shfl_sync(0xffffffffu, incl - bw, bb);
        } else {  // rounding left the target past the piece: its last block of positive weight
            bb = 31 - __clz(static_cast<int>(__ballot_sync(0xffffffffu, bw > 0.0f)) | 1);
            tb = INFINITY;
        }
        // The block's ids: one vector of VEC ids per lane, in order.
        const int v = 32 * bb + lane;
        float xp[VEC], xq[VEC], wv[VEC];
        const bool two = kind == 1;  // the residual's own weights need q_j
        piece_vec_global<Elem>(h.gp, h.len, v, xp);
        if (two) piece_vec_global<Elem>(h.gq, h.len, v, xq);
        float own = 0.0f;
        int lp = -1;
#pragma unroll
        for (int jv = 0; jv < VEC; ++jv) {
            wv[jv] = id_w(xp[jv], two ? xq[jv] : 0.0f);
            if (wv[jv] > 0.0f) lp = v * VEC + jv;
        }
        own = tree_sum<VEC>(wv);
        float c = own;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, c, o);
            if (lane >= o) c += y;
        }
        const unsigned hv = __ballot_sync(0xffffffffu, c > tb);
        int found = -1;
        if (hv) {
            const int hl = __ffs(hv) - 1;
            if (lane == hl) {
                float cum = c - own;
#pragma unroll
                for (int jv = 0; jv < VEC; ++jv) {
                    cum += wv[jv];
                    if (found < 0 && cum > tb) found = v * VEC + jv;
                }
                if (found < 0) found = lp;  // rounding inside the lane
            }
            found = __shfl_sync(0xffffffffu, found, hl);
        }
        if (found < 0) {  // rounding inside the block: its last id of positive weight
            const int lastp = warp_max_int(lp);
            found = lastp >= 0 ? lastp : 32 * bb * VEC;
        }
        token = lo + found;
    }
    // Clear the tail's words for the next call (every piece has been read),
    // write the draw, and finalise the sequence with its last draw.
    uint64_t* dst = a.tpart + static_cast<size_t>(slot) * np * kRecWords;
    for (int kk = lane; kk < np * kRecWords / 2; kk += 32) st_volatile_v2u64(dst + 2 * kk, 0, 0);
    if (lane < kTailWords) st_volatile_u64(a.tdesc + static_cast<size_t>(slot) * kTailWords + lane, 0);
    if (lane == 0) {
        a.tcount[slot] = 0;
        if (t.dest >= 0)
            a.out_tokens[t.dest] = token;
        else
            a.proposals[-1 - t.dest] = token;
        if (atomicAdd(a.seq_done + t.seq, 1) == t.npub - 1) {
            a.seq_done[t.seq] = 0;
            finalize(a);
        }
    }
    return true;
}

// =============================================================================
// Draw kernel workers: every warp takes decision tickets (sequence indices),
// then tail-piece tickets, two pieces in flight at a time, and draws the
// tails whose last piece it finishes
// =============================================================================

// Wait (bounded) for sequence i's ready word: every chunk of the sequence
// reduced and stored by the stream kernel.  The word and the count are
// zeroed for the next call.  False if the wait ran out.
__device__ __forceinline__ bool decide_wait(const VerifyArgs& a, int i, int lane) {
    const uint64_t t0 = global_timer_ns();
    int ok = 1;
    if (lane == 0) {
        while (static_cast<uint32_t>(ld_acquire_u64(a.dready + i) >> 32) != static_cast<uint32_t>(i) + 1u) {
            if (global_timer_ns() - t0 > a.wait_ns) {
                atomicOr(&a.ctl->err, kErrWaitTimeout);
                ok = 0;
                break;
            }
            __nanosleep(128);
        }
        if (ok) {
            st_volatile_u64(a.dready + i, 0);
            a.seq_count[i] = 0;
        }
    }
    __syncwarp();  // every lane reads the partials after lane 0's acquire
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// A warp's first decision ticket (the control block is the previous call's,
// zeroed).
struct FirstDecision {
    unsigned long long ticket;
};

template <typename Elem>
__device__ __forceinline__ FirstDecision first_decision(const VerifyArgs& a, const Tables& tb, int lane) {
    const unsigned long long ndec = tb.batch_bad ? 0ull : static_cast<unsigned long long>(a.num_seqs);
    unsigned long long raw = ndec;
    if (lane == 0 && ndec > 0) raw = atomicAdd(&a.ctl->dclaim, 1ull);
    FirstDecision f;
    f.ticket = __shfl_sync(0xffffffffu, raw, 0);
    return f;
}

// A warp with no piece tickets left draws queued tails: it claims queue
// positions in order and waits for each to be filled (every tail's pieces
// are held by warps that finish them without waiting on a draw).  It stops
// once every sequence is final, or at a claim past the queue's capacity.
template <typename Elem, bool kGum>
__device__ void drawer(const VerifyArgs& a, SmemB& sm, int wi, int n_valid, int lane) {
    for (;;) {
        int raw = 0;
        if (lane == 0) raw = atomicAdd(&a.ctl->draw_claim, 1);
        const int dk = __shfl_sync(0xffffffffu, raw, 0);
        if (dk >= a.n_tail) return;
        const uint64_t t0 = global_timer_ns();
        int slot = -1;
        for (;;) {
            int v = 0, fin = 0;
            if (lane == 0) {
                v = ld_volatile(a.dqueue + dk);
                fin = ld_volatile(&a.ctl->finalized);
            }
            v = __shfl_sync(0xffffffffu, v, 0);
            if (v != 0) {
                slot = v - 1;
                break;
            }
            if (__shfl_sync(0xffffffffu, fin, 0) >= n_valid) return;  // every draw is made
            if (global_timer_ns() - t0 > a.wait_ns) {
                if (lane == 0) atomicOr(&a.ctl->err, kErrWaitTimeout);
                return;
            }
            __nanosleep(128);
        }
        if (lane == 0) a.dqueue[dk] = 0;  // zero again for the next call
        // The tail's descriptor (published before any of its pieces ran).
        uint64_t w = 0;
        for (;;) {
            if (lane < kTailWords) w = ld_volatile_u64(a.tdesc + static_cast<size_t>(slot) * kTailWords + lane);
            if (__all_sync(0xffffffffu, lane >= kTailWords ||
                                            static_cast<uint32_t>(w >> 32) == static_cast<uint32_t>(slot) + 1u))
                break;
            if (global_timer_ns() - t0 > a.wait_ns) {
                if (lane == 0) atomicOr(&a.ctl->err, kErrWaitTimeout);
                return;
            }
        }
        Held hd;
        hd.ticket = 0;
        hd.state = kHeldNone;
        hd.slot = slot;
        hd.k = 0;
        hd.t = decode_tail(w, lane);
        hd.gp = nullptr;
        hd.gq = nullptr;
        hd.len = 0;
        hd.nbytes = 0;
        if (!select_draw<Elem, kGum>(a, sm, wi, hd, lane)) return;
    }
}

template <typename Elem, bool kGum>
__device__ void worker(const VerifyArgs& a, SmemB& sm, int wi, const FirstDecision& first, int lane) {
    const unsigned long long cap = static_cast<unsigned long long>(a.n_tail) * static_cast<unsigned long long>(a.np);
    const unsigned long long ndec = sm.tb.batch_bad ? 0ull : static_cast<unsigned long long>(a.num_seqs);
    const int n_valid = sm.tb.n_valid;
    // Decisions first, each once its sequence's partials are all stored.
    unsigned long long dtk = first.ticket, rawd = 0;
    while (dtk < ndec) {
        if (lane == 0) rawd = atomicAdd(&a.ctl->dclaim, 1ull);
        if (seq_lookup(a, sm.tb, static_cast<int>(dtk)).ok) {
            if (!decide_wait(a, static_cast<int>(dtk), lane)) return;
            const DecPrep pre = decide_prep<Elem>(a, sm.tb, static_cast<int>(dtk), lane);
            decide<Elem>(a, sm.tb, reinterpret_cast<float2*>(sm.buf[wi][0][0]), static_cast<int>(dtk), pre, lane);
            // Every tail slot of the decision is reserved before it counts.
            if (lane == 0) atomic_add_acq_rel(&a.ctl->ddone, 1);
        }
        dtk = __shfl_sync(0xffffffffu, rawd, 0);
    }
    // Two pieces in flight: hc in buffer bc (reduced next), hn in the other.
    Held hc, hn;
    int bc = 0;
    uint32_t pc = 0u, pn = 0u;  // each buffer's barrier phase
    claim_piece(a, hc, cap, lane);
    claim_piece(a, hn, cap, lane);
    uint64_t t_mark = global_timer_ns();
    for (;;) {
        if (hc.state == kHeldWait) try_start<Elem>(a, sm, wi, bc, hc, n_valid, lane);
        if (hn.state == kHeldWait) try_start<Elem>(a, sm, wi, bc ^ 1, hn, n_valid, lane);
        if (hc.state != kHeldLoad) {
            if (hn.state == kHeldLoad || (hc.state == kHeldNone && hn.state != kHeldNone)) {
                const Held tmp = hc;
                hc = hn;
                hn = tmp;
                const uint32_t tp = pc;
                pc = pn;
                pn = tp;
                bc ^= 1;
                if (hc.state != kHeldLoad) continue;
            } else if (hc.state == kHeldNone && hn.state == kHeldNone) {
                drawer<Elem, kGum>(a, sm, wi, n_valid, lane);  // no piece tickets left: draw queued tails
                return;
            } else {
                if (global_timer_ns() - t_mark > a.wait_ns) {
                    if (lane == 0) atomicOr(&a.ctl->err, kErrWaitTimeout);
                    return;
                }
                __nanosleep(64);
                continue;
            }
        }
        // The current piece: wait for its copies; the next ticket for this
        // buffer is claimed while the piece is reduced.
        if (!__all_sync(0xffffffffu, mbar_wait_ns(&sm.bar[wi][bc], pc, kWaitNs))) {
            if (lane == 0) atomicOr(&a.ctl->err, kErrWaitTimeout);
            if (hn.state == kHeldLoad) mbar_wait_ns(&sm.bar[wi][bc ^ 1], pn, kWaitNs);
            return;
        }
        pc ^= 1u;
        unsigned long long raw = 0;
        if (lane == 0) raw = atomicAdd(&a.ctl->claim, 1ull);
        const int cnt = reduce_piece<Elem, kGum>(a, sm.buf[wi][bc][0], sm.buf[wi][bc][1], hc, lane);
        const Held done = hc;
        // The freed buffer starts its next piece before the count comes
        // back: the descriptor's round trip overlaps the count's.
        take_ticket(a, hc, __shfl_sync(0xffffffffu, raw, 0), cap);
        if (hc.state == kHeldWait) try_start<Elem>(a, sm, wi, bc, hc, n_valid, lane);
        // A tail whose pieces are all finished is queued for its draw: the
        // warps that run out of pieces take the draws, so that no piece
        // waits behind one.
        if (lane == 0 && cnt == a.np - 1) st_volatile(a.dqueue + atomicAdd(&a.ctl->draw_tail, 1), done.slot + 1);
        // The other buffer's piece goes next.
        const Held tmp = hc;
        hc = hn;
        hn = tmp;
        const uint32_t tp = pc;
        pc = pn;
        pn = tp;
        bc ^= 1;
        t_mark = global_timer_ns();
    }
}

// =============================================================================
// Kernels
// =============================================================================

// Both kernels' prologue: every CTA counts the valid sequences (the draw
// kernel's exit condition) and the chunks to stream, and checks that the
// offsets never decrease; small batches keep the offsets, temperatures and
// tokens in shared memory.
template <int kThreads>
__device__ __forceinline__ bool load_tables(const VerifyArgs& a, Tables& tb, int tid) {
    if (tid == 0) {
        tb.n_valid = 0;
        tb.units = 0;
    }
    int nv = 0;
    long long nu = 0;
    bool bad = false;
    const bool small = a.num_seqs <= kSmemSeqs;
    for (int i = tid; i < a.num_seqs; i += kThreads) {
        const SeqInfo s = seq_info(a.seq_offsets, a.temperature, i, a.total);
        nv += s.ok ? 1 : 0;
        nu += s.ok ? static_cast<long long>(rows_of(s)) * a.nck : 0;
        const int end = __ldg(a.seq_offsets + i + 1);
        bad = bad || end < s.start;
        if (small) {
            tb.offs[i] = s.start;
            tb.temp[i] = s.T;
            if (i == a.num_seqs - 1) tb.offs[i + 1] = end;
        }
    }
    if (a.total <= kSmemToks)
        for (int r = tid; r < a.total; r += kThreads) tb.tok[r] = __ldg(a.tokens + r);
    __syncthreads();
    if (nv) atomicAdd(&tb.n_valid, nv);
    if (nu) atomicAdd(reinterpret_cast<unsigned long long*>(&tb.units), static_cast<unsigned long long>(nu));
    bad = __syncthreads_or(bad);
    if (tid == 0) {
        tb.batch_bad = bad;
        if (bad) tb.n_valid = 0;
    }
    __syncthreads();
    return bad;
}

template <typename Elem>
__global__ void __launch_bounds__(kThreadsA, kVerifyCtasPerSm) stream_kernel(const VerifyArgs a) {
    extern __shared__ unsigned char smem_raw[];
    SmemA& sm = *reinterpret_cast<SmemA*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~static_cast<uintptr_t>(127));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    pdl_wait();
    // The draw kernel's CTAs may be scheduled from here on, where an SM has
    // room; they run beside this grid and read a sequence's partials once
    // its ready word is published.
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
        fence_mbarrier_init();
    }
    const bool bad = load_tables<kThreadsA>(a, sm.tb, tid);
    if (warp == kProdWarp) {
        if (lane == 0) producer<Elem>(a, sm);
    } else if (warp == kBookWarp) {
        bookkeeper(a, sm, lane);
    } else {
        // This CTA's share of the sequences that are invalid as laid out.
        for (long long i = blockIdx.x + static_cast<long long>(warp) * gridDim.x; i < a.num_seqs;
             i += static_cast<long long>(kCW) * gridDim.x) {
            const SeqInfo s = seq_info(a.seq_offsets, a.temperature, static_cast<int>(i), a.total);
            if (bad || !s.ok) write_invalid(a, static_cast<int>(i), s, lane, -1);
        }
        consumer<Elem>(a, sm, tid, warp, lane);
    }
}

// The draw kernel is compiled once per sampler: each launch carries only
// the code its draws run, which keeps the instruction footprint small.
template <typename Elem, bool kGum>
__global__ void __launch_bounds__(kThreadsB, kCtasPerSmB) draw_kernel(const VerifyArgs a) {
    extern __shared__ unsigned char smem_raw[];
    SmemB& sm = *reinterpret_cast<SmemB*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~static_cast<uintptr_t>(127));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (lane == 0) {
        mbar_init(&sm.bar[warp][0], 1);
        mbar_init(&sm.bar[warp][1], 1);
        fence_mbarrier_init();
    }
    __syncwarp();
    // The draw kernel runs beside the stream kernel: it reads a sequence's
    // partials only after that sequence's ready word (decide_wait).
    load_tables<kThreadsB>(a, sm.tb, tid);
    const FirstDecision first = first_decision<Elem>(a, sm.tb, lane);
    worker<Elem, kGum>(a, sm, warp, first, lane);
    // Every CTA outlasts the stream kernel: the next call's kernels wait for
    // this grid only, and the control block is zeroed below for both.
    pdl_wait();
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
            a.ctl->claim = 0;
            a.ctl->dclaim = 0;
            a.ctl->ddone = 0;
            a.ctl->finalized = 0;
            a.ctl->draw_tail = 0;
            a.ctl->draw_claim = 0;
            a.ctl->exited = 0;
        }
    }
}

static_assert(sizeof(SmemA) + 128 <= 113 * 1024, "two stream CTAs per SM");
static_assert(kCtasPerSmB * (sizeof(SmemB) + 128) <= 227 * 1024, "draw CTAs per SM");
static_assert(kMaxPieces * sizeof(float4) <= 2 * kPieceBytes, "a draw's piece results fit in a worker's first buffer");

template <typename Elem>
cudaError_t launch_verify_t(const VerifyArgs& a, int grid, cudaStream_t stream) {
    const size_t smem_a = sizeof(SmemA) + 128, smem_b = sizeof(SmemB) + 128;
    cudaError_t err = cudaFuncSetAttribute(stream_kernel<Elem>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem_a));
    if (err != cudaSuccess) return err;
    auto* draw = a.sampler == kSamplerGumbel ? draw_kernel<Elem, true> : draw_kernel<Elem, false>;
    err = cudaFuncSetAttribute(draw, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem_b));
    if (err != cudaSuccess) return err;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreadsA);
    cfg.dynamicSmemBytes = smem_a;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    err = cudaLaunchKernelEx(&cfg, stream_kernel<Elem>, a);
    if (err != cudaSuccess) return err;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return cudaErrorUnknown;
    cudaLaunchConfig_t cfg_b = cfg;
    cfg_b.gridDim = dim3(sms * kCtasPerSmB);
    cfg_b.blockDim = dim3(kThreadsB);
    cfg_b.dynamicSmemBytes = smem_b;
    return cudaLaunchKernelEx(&cfg_b, draw, a);
}

}  // namespace

cudaError_t launch_verify(const VerifyArgs& a, int elem_bytes, int grid, cudaStream_t stream) {
    return elem_bytes == 2 ? launch_verify_t<__nv_bfloat16>(a, grid, stream) : launch_verify_t<float>(a, grid, stream);
}

}  // namespace isd
