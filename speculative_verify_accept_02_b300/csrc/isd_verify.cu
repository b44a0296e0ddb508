// The verify step of Introspective Strided Decoding as two kernels
// ("Introspective Diffusion Language Models | Summary", §2 acceptance rate,
// §3.2 strict acceptance, residual correction and bonus token, §3.3 online
// softmax over the vocabulary and a common acceptance path free of
// correction work), optionally with the next stride's proposal draws of the
// fused step (§3.2: one forward verifies and proposes).
//
// stream kernel  every chunk (at most 16 KB) of every row a decision needs:
//                p_k and q_k for k <= L_i (T > 0), or p_1 .. p_{L+1}
//                (T = 0).  Chunks are taken in small batches from a global
//                counter, staged with 1-D bulk copies into a 4-stage ring
//                (mbarrier completion) by one producer thread, and reduced by
//                eight consumer warps to a softmax partial (max, sum) or an
//                argmax per warp; a bookkeeper warp merges the eight and
//                stores the chunk's partial.  Nothing else runs beside the
//                stream: it keeps the HBM busy from its first chunk to its
//                last.
// draw kernel    launched behind it (programmatic dependent launch: its CTAs
//                take the SMs as the stream's retire).  Every warp is a
//                worker:
//                  decisions   by ticket (a sequence index): ratio_k =
//                              min(1, p_k(x_k) / q_k(x_k)), alpha, the accept
//                              prefix (Philox uniforms, one warp ballot;
//                              relaxed acceptance tests min(1, (1 + tau) p/q))
//                              and the emitted prefix; a greedy correction or
//                              bonus.  The draws left are published as tails;
//                  pieces      by ticket: 8 KB of a tail's row or row pair (the
//                              residual max(0, p_j - q_j) of the one rejected
//                              row pair, the final anchor p_{L+1}, or a qnew
//                              row of the fused call), staged in padded shared
//                              memory and reduced, each lane's 128-id block
//                              weight published before the piece's result;
//                  draws       by the worker that finishes a tail's last
//                              piece: by inverse CDF (the piece from the piece
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
constexpr int kStagesV = 4;
constexpr int kRecs = 16;              // record ring between consumers and bookkeeper
constexpr int kGrab = 4;               // units taken from the global counter at once
constexpr int kVecPT = kStageBytes / 16 / kCT;  // 16-byte vectors per consumer thread per stage
constexpr int kWarpsB = 4;             // workers per CTA of the draw kernel
constexpr int kThreadsB = 32 * kWarpsB;
constexpr int kCtasPerSmB = 2;
constexpr int kSmemSeqs = 512;         // batches up to this size keep offsets in shared memory
constexpr int kSmemToks = 1024;        // batches up to this many positions keep their tokens there
constexpr int kPartWords = 4;          // flagged words per piece result
static_assert(kVecPT * 16 * kCT == kStageBytes, "stage split");
// A staged piece row keeps 16 bytes of padding after every 256: a lane that
// reads its own contiguous block of ids then meets no bank conflict.
constexpr int kPieceRow = kPieceBytes + kPieceBytes / 16;
__host__ __device__ constexpr int pad_off(int b) { return b + ((b >> 8) << 4); }

enum : int { kEnd = 0, kUnit = 1 };

struct Desc {
    int kind;
    int seq;
    int slot;        // row slot of the partial: 2 r + {0: p, 1: q}
    int chunk;
    int expect;      // units of the sequence
    int e0;          // first element of the chunk in its row
    int n;           // elements of the chunk
    int nvec;        // 16-byte vectors in shared memory
    int nsm;         // elements of the chunk in shared memory
    int skip;        // elements before e0 in the first vector
    const char* tail;  // global address of the first element not in shared memory
    float c2;        // log2(e) / T, or 0 for an argmax
};

struct Rec {
    int kind, seq, slot, chunk, expect, arg;
    float2 wp[kCW];  // one partial per consumer warp
};

// The batch layout both kernels read: offsets and temperatures of small
// batches, proposed tokens, the valid count.
struct Tables {
    int n_valid;
    int batch_bad;
    int offs[kSmemSeqs + 1];
    float temp[kSmemSeqs];
    int tok[kSmemToks];
};

struct SmemA {
    alignas(128) unsigned char stage[kStagesV][kStageBytes];
    uint64_t full[kStagesV];
    uint64_t empty[kStagesV];
    uint64_t rec_full[kRecs];
    uint64_t rec_empty[kRecs];
    Desc desc[kStagesV];
    Rec rec[kRecs];
    Tables tb;
};

struct SmemB {
    alignas(16) unsigned char piece[kWarpsB][2][kPieceRow];  // each worker's staged piece of p and q
    float4 ppart[kWarpsB][kMaxPieces];                       // each worker's piece results of one draw
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

template <typename Elem>
__device__ void decide(const VerifyArgs& a, const Tables& tb, float2* sblk, int i, int lane) {
    constexpr int E = sizeof(Elem);
    // The stream kernel has completed: every partial of the sequence is in
    // place.
    const SeqInfo s = seq_lookup(a, tb, i);
    const int L = s.len;
    const float T = s.T;
    const float c2 = T > 0.0f ? inv_temp_log2e(T) : 0.0f;
    const int r = s.start + lane;
    const bool mine = lane < L;
    const int x = mine ? (a.total <= kSmemToks ? tb.tok[r] : __ldg(a.tokens + r)) : 0;
    if (__any_sync(0xffffffffu, mine && (x < 0 || x >= a.vocab))) {
        write_invalid(a, i, s, lane, -1);
        if (lane == 0) finalize(a);
        return;
    }
    const bool stall = i == a.stall_seq;
    // A T > 0 sequence always makes one draw after its decision: its queue
    // slot is reserved now, so that the round trip overlaps the loads below.
    int tslot = 0;
    if (T > 0.0f && lane == 0 && !stall) tslot = atomicAdd(&a.ctl->tail_reserve, 1);
    // The sequence's partials are one contiguous block, [2 L rows][nck]: it
    // is staged in this warp's shared buffer in one round trip, together
    // with the proposed tokens' logits, when it fits.
    const float2* blk = a.part + static_cast<size_t>(2 * s.start) * a.nck;
    const int nblk = 2 * L * a.nck;
    const bool staged = nblk * static_cast<int>(sizeof(float2)) <= 2 * kPieceRow;
    if (staged)
        for (int v = lane; v < nblk / 2; v += 32) cp_async16(sblk + 2 * v, blk + 2 * v);
    float zp = 0.0f, zq = 0.0f;
    if (mine && T > 0.0f) {  // the proposed token's logits, from rows read moments ago
        zp = load_elem<Elem>(a.p + static_cast<int64_t>(r + i) * a.ldp_bytes + static_cast<size_t>(x) * E);
        zq = load_elem<Elem>(a.q + static_cast<int64_t>(r) * a.ldq_bytes + static_cast<size_t>(x) * E);
    }
    // The accept uniform does not depend on the loads: it is drawn while
    // they are in flight.
    const float u_acc = (mine && T > 0.0f) ? decision_uniform(a.seed, a.offset, i, lane + 1, kTagAccept) : 0.0f;
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
    if (stall) return;  // check hook: nothing is published, the sequence never completes
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
// group g (8 lanes, one per consumer warp) handles record r + g.
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
        const int kind = rc.kind, rslot = rc.slot, chunk = rc.chunk, arg = rc.arg;
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
        if (g < n_real && wl == 0)
            a.part[static_cast<size_t>(rslot) * a.nck + chunk] = arg ? make_float2(Ma, __int_as_float(Ia))
                                                                     : make_float2(Mm, Sm);
        __syncwarp();
        r += nb;
        if (end_mask) break;
    }
}

// =============================================================================
// Producer thread (stream kernel): streams chunks into the stage ring
// =============================================================================

__device__ __forceinline__ int acquire_stage(SmemA& sm, long long n, int* err) {
    const int stage = static_cast<int>(n % kStagesV);
    const uint32_t parity = (static_cast<uint32_t>(n / kStagesV) & 1u) ^ 1u;
    if (!mbar_wait_ns(&sm.empty[stage], parity, kWaitNs)) {
        atomicOr(err, kErrWaitTimeout);
        return -1;
    }
    return stage;
}

template <typename Elem>
__device__ void producer(const VerifyArgs& a, SmemA& sm) {
    constexpr int E = sizeof(Elem);
    long long n = 0;  // stages issued
    bool ok = true;
    if (!sm.tb.batch_bad) {
        // Units in sequence order: sequence i owns [base, base + units);
        // within it, row index ri in [0, rows_of), chunk c in [0, nck).  A
        // batch of kGrab units is taken from the global counter one batch
        // ahead of its use, so a CTA that falls behind takes fewer.
        int i = -1;
        long long base = 0, units = 0;
        SeqInfo s{};
        float c2 = 0.0f;
        unsigned long long next = atomicAdd(&a.ctl->grab, static_cast<unsigned long long>(kGrab));
        unsigned long long cur = 0, cur_end = 0;
        while (ok) {
            if (cur == cur_end) {
                cur = next;
                cur_end = next + kGrab;
                next = atomicAdd(&a.ctl->grab, static_cast<unsigned long long>(kGrab));
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
            const int stage = acquire_stage(sm, n, &a.ctl->err);
            if (stage < 0) {
                ok = false;
                break;
            }
            Desc& d = sm.desc[stage];
            d.kind = kUnit;
            d.seq = i;
            d.slot = slot;
            d.chunk = c;
            d.expect = static_cast<int>(units);
            d.e0 = e0;
            d.n = nel;
            d.nvec = pc.bytes >> 4;
            d.nsm = pc.nsm;
            d.skip = pc.skip;
            d.tail = pc.tail;
            d.c2 = c2;
            if (pc.bytes > 0) {
                mbar_arrive_expect_tx(&sm.full[stage], static_cast<uint32_t>(pc.bytes));
                bulk_copy_g2s(sm.stage[stage], reinterpret_cast<const void*>(pc.lo), static_cast<uint32_t>(pc.bytes),
                              &sm.full[stage]);
            } else {
                mbar_arrive(&sm.full[stage]);
            }
            ++n;
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

// Hand this warp's partial of a unit to the bookkeeper.
__device__ __forceinline__ void push_record(const VerifyArgs& a, SmemA& sm, long long& nrec, int warp, int lane,
                                            float2 part, int kind, int seq, int slot, int chunk, int expect,
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
            rc.slot = slot;
            rc.chunk = chunk;
            rc.expect = expect;
            rc.arg = arg;
        }
        mbar_arrive(&sm.rec_full[rs]);
    }
    __syncwarp();
}

template <typename Elem>
__device__ __forceinline__ void unit_stage(const VerifyArgs& a, SmemA& sm, int stage, const Desc& d, int tid,
                                           int warp, int lane, long long& nrec) {
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
    float2 part;
    if (c2 > 0.0f) {
        float M = -INFINITY, S = 0.0f;
        if (cm != -INFINITY) {
            const float mc = cm * c2;
            const uint64_t C2 = pack_f2(c2, c2), NMC = pack_f2(-mc, -mc);
            uint64_t acc0 = 0, acc1 = 0;
#pragma unroll
            for (int j = 0; j < kVecPT * 4; j += 2) {
                if constexpr (kBf16) {
                    float y0, y1, y2, y3;
                    unpack_f2(fma_f2(pack_f2(bf16lo(w[j]), bf16hi(w[j])), C2, NMC), y0, y1);
                    unpack_f2(fma_f2(pack_f2(bf16lo(w[j + 1]), bf16hi(w[j + 1])), C2, NMC), y2, y3);
                    acc0 = add_f2(acc0, pack_f2(ex2_approx(y0), ex2_approx(y1)));
                    acc1 = add_f2(acc1, pack_f2(ex2_approx(y2), ex2_approx(y3)));
                } else {
                    float y0, y1;
                    unpack_f2(fma_f2(pack_f2(__uint_as_float(w[j]), __uint_as_float(w[j + 1])), C2, NMC), y0, y1);
                    if (j & 2)
                        acc1 = add_f2(acc1, pack_f2(ex2_approx(y0), ex2_approx(y1)));
                    else
                        acc0 = add_f2(acc0, pack_f2(ex2_approx(y0), ex2_approx(y1)));
                }
            }
            if (tv != -INFINITY) acc1 = add_f2(acc1, pack_f2(soft_w(tv, c2, mc), 0.0f));
            float s0, s1, s2, s3;
            unpack_f2(acc0, s0, s1);
            unpack_f2(acc1, s2, s3);
            M = mc;
            S = (s0 + s1) + (s2 + s3);
        }
        warp_merge_mc(M, S);
        part = make_float2(M, S);
    } else {
        // First position of the maximum in this thread's (ascending) elements.
        constexpr int kPer = kBf16 ? 8 : 4;
        int idx = INT_MAX;
        if (cm != -INFINITY) {  // a chunk of -inf alone has no maximum to offer
            if (tv == cm) idx = d.nsm + tid;
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
        }
        float M = cm;
        int I = idx == INT_MAX ? INT_MAX : d.e0 + idx;
        warp_merge_arg(M, I);
        part = make_float2(M, __int_as_float(I));
    }
    push_record(a, sm, nrec, warp, lane, part, kUnit, d.seq, d.slot, d.chunk, d.expect, c2 > 0.0f ? 0 : 1);
}

template <typename Elem>
__device__ void consumer(const VerifyArgs& a, SmemA& sm, int tid, int warp, int lane) {
    long long nrec = 0;
    for (long long n = 0;; ++n) {
        const int stage = static_cast<int>(n % kStagesV);
        const uint32_t parity = static_cast<uint32_t>(n / kStagesV) & 1u;
        if (!__all_sync(0xffffffffu, mbar_wait_ns(&sm.full[stage], parity, kDrainWaitNs + kWaitNs))) {
            if (lane == 0) atomicOr(&a.ctl->err, kErrWaitTimeout);
            break;
        }
        const Desc d = sm.desc[stage];
        if (d.kind == kEnd) break;
        unit_stage<Elem>(a, sm, stage, d, tid, warp, lane, nrec);
    }
    // Tell the bookkeeper there is no more work (a record of kind kEnd).
    push_record(a, sm, nrec, warp, lane, make_float2(0.0f, 0.0f), kEnd, 0, 0, 0, 0, 0);
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

// Stage elements [0, n) of a piece of one or two rows (from gp, and gq when
// `two`) in shared memory (padded rows, pad_off), every load in flight at
// once: 16-byte cp.async where both rows allow them, the elements left one
// by one.
template <typename Elem>
__device__ __forceinline__ void stage_piece(unsigned char* sp, unsigned char* sq, const char* gp, const char* gq,
                                            int n, bool two, int lane) {
    constexpr int E = sizeof(Elem), VEC = 16 / E;
    const bool v16 = aligned16(gp) && (!two || aligned16(gq));
    const int nv16 = v16 ? (n * E) >> 4 : 0;
    for (int v = lane; v < nv16; v += 32) {
        cp_async16(sp + pad_off(16 * v), gp + 16 * v);
        if (two) cp_async16(sq + pad_off(16 * v), gq + 16 * v);
    }
    using Raw = typename std::conditional<E == 2, uint16_t, uint32_t>::type;
    for (int e = nv16 * VEC + lane; e < n; e += 32) {
        *reinterpret_cast<Raw*>(sp + pad_off(e * E)) = reinterpret_cast<const Raw*>(gp)[e];
        if (two) *reinterpret_cast<Raw*>(sq + pad_off(e * E)) = reinterpret_cast<const Raw*>(gq)[e];
    }
    cp_async_wait_all();
    __syncwarp();
}

// Ids e .. e + 16/E - 1 of a staged (padded) piece row, -inf past n.
template <typename Elem>
__device__ __forceinline__ void staged_vec(const unsigned char* st, int e, int n, float x[16 / sizeof(Elem)]) {
    constexpr int E = sizeof(Elem), VEC = 16 / E;
    const uint4 v = *reinterpret_cast<const uint4*>(st + pad_off(e * E));
#pragma unroll
    for (int jv = 0; jv < VEC; ++jv) x[jv] = e + jv < n ? vec_elem<E>(v, jv) : -INFINITY;
}

// One piece (ids [k ps, k ps + ps) of the tail's row or row pair), staged in
// this worker's buffer, then reduced.  Lane l takes the contiguous block of
// ids [l q, l q + q), q = ps / 32, and publishes its block's weight (inverse
// CDF), so that a draw can find its block without scanning the piece.  The
// piece's result follows as four flagged words:
//   inverse CDF, residual:  (sum of max(0, p - q), sum of p)
//   inverse CDF, softmax:   (mc, sum exp2(x c2 - mc)), mc = the piece's largest logit times c2
//   argmax (T = 0):         (max, lowest id)
//   Gumbel-max:             (best score, its id, best score of p alone, its id)
// where a Gumbel score is log2 w_v - log2(-ln u_v); the last pair is the
// fallback for a residual that rounds to zero everywhere.  Returns true for
// the piece that completes its tail.
template <typename Elem>
__device__ bool run_piece(const VerifyArgs& a, unsigned char* sp, unsigned char* sq, const Tail& t, int slot, int k,
                          int lane) {
    constexpr int E = sizeof(Elem), VEC = 16 / E;
    constexpr int kPerLane = kPieceBytes / E / 32;
    const int e0 = k * a.ps;
    const int n = min(a.ps, a.vocab - e0);
    const bool res = t.mode == kTailRes;
    const bool gum = a.sampler == kSamplerGumbel && t.mode != kTailArg;
    stage_piece<Elem>(sp, sq, tail_prow<Elem>(a, t) + static_cast<size_t>(e0) * E,
                      a.q + static_cast<int64_t>(t.qrow) * a.ldq_bytes + static_cast<size_t>(e0) * E, n, res, lane);
    const int b = lane * kPerLane;  // this lane's block of ids
    uint32_t out[kPartWords] = {0, 0, 0, 0};
    if (gum || t.mode == kTailArg) {
        float best = -INFINITY, best_p = -INFINITY;
        int bid = INT_MAX, bid_p = INT_MAX;
        for (int j = 0; j < kPerLane; j += VEC) {
            const int e = b + j;
            if (e >= n) break;
            float xp[VEC], xq[VEC];
            staged_vec<Elem>(sp, e, n, xp);
            if (res) staged_vec<Elem>(sq, e, n, xq);
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
                            const float w = resid_w(xp[jv], xq[jv], t.c2, t.nz0, t.nz1, pv);
                            lw = w > 0.0f ? lg2_approx(w) : -INFINITY;
                            lpw = pv > 0.0f ? lg2_approx(pv) : -INFINITY;
                        } else {
                            lw = xp[jv] * t.c2;
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
            } else {  // argmax: the first maximum is kept
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
        // Inverse CDF: the block's weight and the piece's sums, independent
        // exponentials summed as small trees.
        float mc = 0.0f;
        if (!res) {  // the softmax partial's reference: the piece's largest logit times c2
            float m = -INFINITY;
#pragma unroll 4
            for (int j = 0; j < kPerLane; j += VEC) {
                float xp[VEC];
                staged_vec<Elem>(sp, b + j, n, xp);
#pragma unroll
                for (int jv = 0; jv < VEC; ++jv) m = fmaxf(m, xp[jv]);
            }
            m = warp_max(m);
            mc = m == -INFINITY ? -INFINITY : m * t.c2;
        }
        float bw = 0.0f, bp = 0.0f;
        if (res || mc != -INFINITY) {
#pragma unroll 2
            for (int j = 0; j < kPerLane; j += VEC) {
                float xp[VEC], w[VEC], pv[VEC];
                staged_vec<Elem>(sp, b + j, n, xp);
                if (res) {
                    float xq[VEC];
                    staged_vec<Elem>(sq, b + j, n, xq);
#pragma unroll
                    for (int jv = 0; jv < VEC; ++jv) w[jv] = resid_w(xp[jv], xq[jv], t.c2, t.nz0, t.nz1, pv[jv]);
                    bp += tree_sum<VEC>(pv);
                } else {
#pragma unroll
                    for (int jv = 0; jv < VEC; ++jv) w[jv] = soft_w(xp[jv], t.c2, mc);
                }
                bw += tree_sum<VEC>(w);
            }
        }
        a.tbsum[(static_cast<size_t>(slot) * a.np + k) * 32 + lane] = bw;
        if (res) {
            out[0] = __float_as_uint(warp_sum(bw));
            out[1] = __float_as_uint(warp_sum(bp));
        } else {
            out[0] = __float_as_uint(mc);
            out[1] = __float_as_uint(mc == -INFINITY ? 0.0f : warp_sum(bw));
        }
        __syncwarp();
        if (lane == 0) __threadfence();  // the block weights are visible before the result
    }
    int last = 0;
    if (lane == 0) {
        const uint32_t f = static_cast<uint32_t>(slot) + 1u;
        uint64_t* dst = a.tpart + (static_cast<size_t>(slot) * a.np + k) * kPartWords;
        st_volatile_v2u64(dst, flagged(f, out[0]), flagged(f, out[1]));
        st_volatile_v2u64(dst + 2, flagged(f, out[2]), flagged(f, out[3]));
        // The results carry their flags, so the count needs no ordering.
        last = atomicAdd(a.tcount + slot, 1) == a.np - 1;
    }
    return __shfl_sync(0xffffffffu, last, 0) != 0;
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

// Inverse-CDF position of `target` in the running weight of a staged piece
// of `len` ids (weights w(xp, xq) of its staged, padded p and q logits), in
// vocabulary order.  Lane l sums ids [l q, l q + q) from 16-byte vectors;
// the lane whose block holds the target is then walked by the whole warp, a
// few ids per lane.  Rounding that leaves the target past the block's end
// gives the block's last id of positive weight, past every weight the
// piece's last one.
template <typename Elem, typename F>
__device__ __forceinline__ int piece_icdf(const unsigned char* sp, const unsigned char* sq, bool two, int len,
                                          float target, const F& w, int lane) {
    constexpr int E = sizeof(Elem), VEC = 16 / E;
    constexpr int kPerLane = kPieceBytes / E / 32;
    constexpr int kSub = kPerLane / 32;
    const int b = lane * kPerLane;
    float own = 0.0f;
    int lp = -1;
    // A whole vector's weights at a time, independent of each other (ids
    // past the piece read as -inf, weight 0), summed as a small tree.
#pragma unroll 2
    for (int j = 0; j < kPerLane; j += VEC) {
        const int e = b + j;
        const uint4 vp = *reinterpret_cast<const uint4*>(sp + pad_off(e * E));
        const uint4 vq = two ? *reinterpret_cast<const uint4*>(sq + pad_off(e * E)) : make_uint4(0, 0, 0, 0);
        float wv[VEC];
#pragma unroll
        for (int jv = 0; jv < VEC; ++jv) {
            const bool in = e + jv < len;
            wv[jv] = w(in ? vec_elem<E>(vp, jv) : -INFINITY, in ? vec_elem<E>(vq, jv) : -INFINITY);
        }
#pragma unroll
        for (int jv = 0; jv < VEC; ++jv)
            if (wv[jv] > 0.0f) lp = e + jv;
        own += tree_sum<VEC>(wv);
    }
    float incl = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    const unsigned hit = __ballot_sync(0xffffffffu, b < len && incl > target);
    int found = -1;
    if (hit) {
        const int owner = __ffs(hit) - 1;
        const float before = __shfl_sync(0xffffffffu, incl - own, owner);
        const int olp = __shfl_sync(0xffffffffu, lp, owner);  // the block's last id of positive weight
        const int ob = owner * kPerLane + lane * kSub;          // this lane's ids of the owner's block
        float sub = 0.0f;
#pragma unroll
        for (int e = 0; e < kSub; ++e)
            if (ob + e < len)
                sub += w(load_elem<Elem>(sp + pad_off((ob + e) * E)),
                         two ? load_elem<Elem>(sq + pad_off((ob + e) * E)) : 0.0f);
        float c = sub;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, c, o);
            if (lane >= o) c += y;
        }
        const unsigned h = __ballot_sync(0xffffffffu, ob < len && before + c > target);
        if (h) {
            const int hl = __ffs(h) - 1;
            if (lane == hl) {
                float cum = before + c - sub;
                int last = -1;
#pragma unroll
                for (int e = 0; e < kSub; ++e) {
                    if (found < 0 && ob + e < len) {
                        const float x = w(load_elem<Elem>(sp + pad_off((ob + e) * E)),
                                          two ? load_elem<Elem>(sq + pad_off((ob + e) * E)) : 0.0f);
                        cum += x;
                        if (x > 0.0f) last = ob + e;
                        if (cum > target) found = ob + e;
                    }
                }
                if (found < 0) found = last >= 0 ? last : olp;  // rounding inside the lane
            }
            found = __shfl_sync(0xffffffffu, found, hl);
        } else {
            found = olp;  // rounding inside the block
        }
    }
    if (found < 0) {
        const int last = warp_max_int(lp);
        found = last >= 0 ? last : 0;
    }
    return found;
}

// The draw of tail `slot`, by the worker whose piece completed it: reads every
// piece result (all counted, their flagged words land moments later at
// most), draws, writes the token, and clears the tail's words and count for
// the next call.  False if a wait ran out.
template <typename Elem>
__device__ bool select_draw(const VerifyArgs& a, unsigned char* sp, unsigned char* sq, float4* pr, const Tail& t,
                            int slot, int lane) {
    constexpr int E = sizeof(Elem);
    const int np = a.np;
    const uint32_t f = static_cast<uint32_t>(slot) + 1u;
    const uint64_t* src = a.tpart + static_cast<size_t>(slot) * np * kPartWords;
    const bool gum = a.sampler == kSamplerGumbel && t.mode != kTailArg;
    // The draw's uniform, while the results are on their way.
    const float rnd = (gum || t.mode == kTailArg) ? 0.0f : decision_uniform(a.seed, a.offset, t.seq, t.pos, t.tag);
    // Wait for every piece: each lane polls pieces lane, lane + 32, ...
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        bool mine = true;
        for (int kp = lane; kp < np; kp += 32) {
            uint64_t w0, w1, w2, w3;
            ld_volatile_v2u64(src + static_cast<size_t>(kp) * kPartWords, w0, w1);
            ld_volatile_v2u64(src + static_cast<size_t>(kp) * kPartWords + 2, w2, w3);
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
        // piece, then its id within the piece, every sum in vocabulary order.
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
        const int lo = chosen * a.ps;
        const int len = min(a.ps, a.vocab - lo);
        const bool res = t.mode == kTailRes;
        const char* gp = tail_prow<Elem>(a, t) + static_cast<size_t>(lo) * E;
        const char* gq = a.q + static_cast<int64_t>(t.qrow) * a.ldq_bytes + static_cast<size_t>(lo) * E;
        if (kind == 2) {
            // A residual that rounded to zero everywhere draws from p_j: no
            // block weights of p were kept, so the piece is staged and
            // scanned whole (a path that rounding alone can reach).
            stage_piece<Elem>(sp, sq, gp, gq, len, res, lane);
            const DrawW id_w{kind, t.c2, MC, t.nz0, t.nz1};
            token = lo + piece_icdf<Elem>(sp, sq, res, len, tloc, id_w, lane);
        } else {
            // The block: its weight per lane, published before the piece's
            // result (acquired by the fence), in the piece's own scale.
            __threadfence();
            const float mc_k = soft ? pr[chosen].x : 0.0f;
            const float tpiece = soft ? tloc * ex2_approx(MC - mc_k) : tloc;
            const float bw = __ldcg(a.tbsum + (static_cast<size_t>(slot) * np + chosen) * 32 + lane);
            constexpr int kPerLane = kPieceBytes / E / 32;
            constexpr int kSub = kPerLane / 32;
            float incl = bw;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            const unsigned hit = __ballot_sync(0xffffffffu, incl > tpiece);
            int bb;
            float tb;
            if (hit) {
                bb = __ffs(hit) - 1;
                tb = tpiece - __shfl_sync(0xffffffffu, incl - bw, bb);
            } else {  // rounding left the target past the piece: its last block of positive weight
                bb = 31 - __clz(static_cast<int>(__ballot_sync(0xffffffffu, bw > 0.0f)) | 1);
                tb = INFINITY;
            }
            // The block's ids straight from the rows: kSub per lane, in order.
            const DrawW id_w{kind, t.c2, soft ? mc_k : MC, t.nz0, t.nz1};
            const int ib = bb * kPerLane + lane * kSub;  // this lane's ids in the piece
            float wv[kSub];
            float own = 0.0f;
            int lp = -1;
#pragma unroll
            for (int e = 0; e < kSub; ++e) {
                const bool in = ib + e < len;
                const float xp = in ? load_elem<Elem>(gp + static_cast<size_t>(ib + e) * E) : -INFINITY;
                const float xq = (in && res) ? load_elem<Elem>(gq + static_cast<size_t>(ib + e) * E) : -INFINITY;
                wv[e] = id_w(xp, xq);
                own += wv[e];
                if (wv[e] > 0.0f) lp = ib + e;
            }
            float c = own;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, c, o);
                if (lane >= o) c += y;
            }
            const unsigned h = __ballot_sync(0xffffffffu, c > tb);
            int found = -1;
            if (h) {
                const int hl = __ffs(h) - 1;
                if (lane == hl) {
                    float cum = c - own;
#pragma unroll
                    for (int e = 0; e < kSub; ++e) {
                        cum += wv[e];
                        if (found < 0 && cum > tb) found = ib + e;
                    }
                    if (found < 0) found = lp;  // rounding inside the lane
                }
                found = __shfl_sync(0xffffffffu, found, hl);
            }
            if (found < 0) {  // rounding inside the block: its last id of positive weight
                const int lastp = warp_max_int(lp);
                found = lastp >= 0 ? lastp : bb * kPerLane;
            }
            token = lo + found;
        }
    }
    // Clear the tail's words for the next call (every piece has been read),
    // write the draw, and finalise the sequence with its last draw.
    uint64_t* dst = a.tpart + static_cast<size_t>(slot) * np * kPartWords;
    for (int kk = lane; kk < np; kk += 32) {
        st_volatile_v2u64(dst + static_cast<size_t>(kk) * kPartWords, 0, 0);
        st_volatile_v2u64(dst + static_cast<size_t>(kk) * kPartWords + 2, 0, 0);
    }
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

// A worker holds one decision ticket (a sequence index: sequences complete
// roughly in index order, as the units are dealt) and one tail-piece ticket
// (a queue slot and a piece), and serves whichever comes ready first.
// =============================================================================
// Draw kernel workers: every warp takes decision tickets (sequence indices),
// then tail-piece tickets, and draws the tails whose last piece it finishes
// =============================================================================

template <typename Elem>
__device__ void worker(const VerifyArgs& a, SmemB& sm, int wi, int lane) {
    const unsigned long long cap = static_cast<unsigned long long>(a.n_tail) * static_cast<unsigned long long>(a.np);
    const unsigned long long ndec = sm.tb.batch_bad ? 0ull : static_cast<unsigned long long>(a.num_seqs);
    const int n_valid = sm.tb.n_valid;
    unsigned char* sp = sm.piece[wi][0];
    unsigned char* sq = sm.piece[wi][1];
    unsigned long long raw = 0, rawd = 0;
    if (lane == 0) rawd = ndec > 0 ? atomicAdd(&a.ctl->dclaim, 1ull) : ndec;
    unsigned long long dtk = __shfl_sync(0xffffffffu, rawd, 0);
    // Decisions first: every sequence is ready, its partials complete.
    while (dtk < ndec) {
        if (lane == 0) rawd = atomicAdd(&a.ctl->dclaim, 1ull);
        if (seq_lookup(a, sm.tb, static_cast<int>(dtk)).ok)
            decide<Elem>(a, sm.tb, reinterpret_cast<float2*>(sp), static_cast<int>(dtk), lane);
        dtk = __shfl_sync(0xffffffffu, rawd, 0);
    }
    if (lane == 0) raw = cap > 0 ? atomicAdd(&a.ctl->claim, 1ull) : cap;
    unsigned long long ticket = __shfl_sync(0xffffffffu, raw, 0);
    uint64_t t_mark = global_timer_ns();
    for (;;) {
        const bool have = ticket < cap;
        const int slot = have ? static_cast<int>(ticket / static_cast<unsigned long long>(a.np)) : 0;
        const int k = have ? static_cast<int>(ticket % static_cast<unsigned long long>(a.np)) : 0;
        // One round trip: the held ticket's descriptor and the completion count.
        uint64_t w = 0;
        if (have && lane < kTailWords) w = ld_volatile_u64(a.tdesc + static_cast<size_t>(slot) * kTailWords + lane);
        int fin = 0;
        if (lane == 31) fin = ld_volatile(&a.ctl->finalized);
        const bool ready = have && __all_sync(0xffffffffu, lane >= kTailWords ||
                                                               static_cast<uint32_t>(w >> 32) == static_cast<uint32_t>(slot) + 1u);
        if (ready) {
            const Tail t = decode_tail(w, lane);
            // The next ticket is claimed now; its round trip overlaps the piece.
            if (lane == 0) raw = atomicAdd(&a.ctl->claim, 1ull);
            if (run_piece<Elem>(a, sp, sq, t, slot, k, lane) && !select_draw<Elem>(a, sp, sq, sm.ppart[wi], t, slot, lane))
                return;
            ticket = __shfl_sync(0xffffffffu, raw, 0);
            t_mark = global_timer_ns();
            continue;
        }
        fin = __shfl_sync(0xffffffffu, fin, 31);
        if (fin >= n_valid) return;  // every sequence is final
        if (global_timer_ns() - t_mark > a.wait_ns) {
            if (lane == 0) atomicOr(&a.ctl->err, kErrWaitTimeout);
            return;
        }
        __nanosleep(64);
    }
}

// =============================================================================
// Kernels
// =============================================================================

// Both kernels' prologue: every CTA counts the valid sequences (the draw
// kernel's exit condition) and checks that the offsets never decrease; small
// batches keep the offsets, temperatures and tokens in shared memory.
template <int kThreads>
__device__ __forceinline__ bool load_tables(const VerifyArgs& a, Tables& tb, int tid) {
    if (tid == 0) tb.n_valid = 0;
    int nv = 0;
    bool bad = false;
    const bool small = a.num_seqs <= kSmemSeqs;
    for (int i = tid; i < a.num_seqs; i += kThreads) {
        const SeqInfo s = seq_info(a.seq_offsets, a.temperature, i, a.total);
        nv += s.ok ? 1 : 0;
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
    // The draw kernel's CTAs may be scheduled as soon as SMs free up; they
    // wait for this grid to complete before reading anything it writes.
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

template <typename Elem>
__global__ void __launch_bounds__(kThreadsB, kCtasPerSmB) draw_kernel(const VerifyArgs a) {
    extern __shared__ unsigned char smem_raw[];
    SmemB& sm = *reinterpret_cast<SmemB*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~static_cast<uintptr_t>(127));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    pdl_wait();  // the stream kernel has completed and its partials are visible
    load_tables<kThreadsB>(a, sm.tb, tid);
    worker<Elem>(a, sm, warp, lane);
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
            a.ctl->finalized = 0;
            a.ctl->exited = 0;
        }
    }
}

static_assert(sizeof(SmemA) + 128 <= 113 * 1024, "two stream CTAs per SM");
static_assert(kCtasPerSmB * (sizeof(SmemB) + 128) <= 227 * 1024, "draw CTAs per SM");

template <typename Elem>
cudaError_t launch_verify_t(const VerifyArgs& a, int grid, cudaStream_t stream) {
    const size_t smem_a = sizeof(SmemA) + 128, smem_b = sizeof(SmemB) + 128;
    cudaError_t err = cudaFuncSetAttribute(stream_kernel<Elem>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem_a));
    if (err != cudaSuccess) return err;
    err = cudaFuncSetAttribute(draw_kernel<Elem>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem_b));
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
    return cudaLaunchKernelEx(&cfg_b, draw_kernel<Elem>, a);
}

}  // namespace

cudaError_t launch_verify(const VerifyArgs& a, int elem_bytes, int grid, cudaStream_t stream) {
    return elem_bytes == 2 ? launch_verify_t<__nv_bfloat16>(a, grid, stream) : launch_verify_t<float>(a, grid, stream);
}

}  // namespace isd
