// The propose step of Introspective Strided Decoding as one kernel
// ("Introspective Diffusion Language Models | Summary", §3.2: the mask
// positions of a forward give the next stride's proposals; §3.3: argmax
// proposals at T = 0).
//
// Work is the rows whose proposals are kept (every CTA lists them from the
// batch layout in shared memory), each cut into runs of consecutive chunks of
// at most 16 KB -- as many runs as keep every CTA busy, a whole row per CTA
// once rows outnumber CTAs -- dealt round-robin.  A CTA streams its run with
// 16-byte vector loads, the next chunk in flight while each warp reduces its
// share of the current one to a softmax partial (max * log2(e)/T, sum of exp2
// relative to it) or an exact argmax (max, lowest id), without block
// barriers.  The CTA that completes a row draws its proposal: the chunk by
// inverse CDF over the row's chunk partials, then an in-order scan of that one
// chunk staged in shared memory.  No CTA ever waits for another.
#include <climits>

#include "isd_device.cuh"
#include "isd_internal.h"

namespace isd {
namespace {

constexpr int kPT = 512;              // threads per CTA
constexpr int kPW = kPT / 32;
constexpr int kPSeqs = 512;           // batches up to this size keep their layout in shared memory
constexpr int kPVec = kStageBytes / 16 / kPT;  // 16-byte vectors per thread per chunk (2)

struct PropShared {
    alignas(16) unsigned char chunk[kStageBytes];  // the chosen chunk of a row being drawn
    float2 part[kMaxProposeChunks];                // that row's chunk partials
    float2 wpart[kMaxProposeChunks][kPW];          // per-warp partials of the chunks of a piece
    int offs[kPSeqs + 1];
    float temp[kPSeqs];
    int acc[kPSeqs];
    unsigned char draw[kPSeqs];
    int pref[kPSeqs + 1];  // drawn rows of the sequences before i
    int wsum[kPW];
    int item_i, item_r;    // large batches: the current item's sequence and row (-1: skip)
    float red_m[kPW];
    float red_s[kPW];
    int red_i[kPW];
    int red_j[kPW];
    int bad;
    int last;
    int sel_chunk;
    float sel_t;
    float sel_mc;
};

template <typename Elem>
__device__ __forceinline__ float raw_elem(const unsigned char* p) {
    if constexpr (sizeof(Elem) == 2)
        return __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(p)) << 16);
    else
        return *reinterpret_cast<const float*>(p);
}

// Elements [e0, e0 + n) of a row: the 16-byte aligned interior is loaded as
// vectors, the unaligned head and tail (fewer than 16 bytes each) element by
// element.
struct Span {
    uintptr_t sb;    // address of element e0
    uintptr_t lo;    // first aligned byte of the interior
    int head;        // elements before lo
    int nvec;        // 16-byte vectors of the interior
    int tail;        // elements after the interior
};

template <int E>
__device__ __forceinline__ Span make_span(const char* row, int e0, int n) {
    Span sp;
    sp.sb = reinterpret_cast<uintptr_t>(row) + static_cast<uintptr_t>(e0) * E;
    const uintptr_t eb = sp.sb + static_cast<uintptr_t>(n) * E;
    const uintptr_t lo = (sp.sb + 15) & ~static_cast<uintptr_t>(15), hi = eb & ~static_cast<uintptr_t>(15);
    if (lo < hi) {
        sp.lo = lo;
        sp.head = static_cast<int>((lo - sp.sb) / E);
        sp.nvec = static_cast<int>((hi - lo) / 16);
        sp.tail = static_cast<int>((eb - hi) / E);
    } else {
        sp.lo = sp.sb;
        sp.head = n;
        sp.nvec = 0;
        sp.tail = 0;
    }
    return sp;
}

// Warp-wide merge of (mc, s) softmax partials; every lane gets the result.
__device__ __forceinline__ void warp_merge_mc2(float& M, float& S) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) merge_mc(M, S, __shfl_xor_sync(0xffffffffu, M, o), __shfl_xor_sync(0xffffffffu, S, o));
}

// Block-wide (max, lowest id); every thread gets the result.
__device__ void block_merge_arg(PropShared& sh, float& M, int& I) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) merge_argmax(M, I, __shfl_xor_sync(0xffffffffu, M, o), __shfl_xor_sync(0xffffffffu, I, o));
    if (lane == 0) {
        sh.red_m[warp] = M;
        sh.red_i[warp] = I;
    }
    __syncthreads();
    M = lane < kPW ? sh.red_m[lane] : -INFINITY;
    I = lane < kPW ? sh.red_i[lane] : INT_MAX;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) merge_argmax(M, I, __shfl_xor_sync(0xffffffffu, M, o), __shfl_xor_sync(0xffffffffu, I, o));
    __syncthreads();
}

// Whether sequence i's proposals are drawn (shared-memory layout or global).
struct PSeq {
    int start, len;
    float T;
    bool draw;
};

__device__ __forceinline__ PSeq pseq(const ProposeArgs& a, const PropShared& sh, int i) {
    PSeq q;
    int end;
    if (a.num_seqs <= kPSeqs) {  // decided once per CTA in the prologue
        q.start = sh.offs[i];
        q.len = sh.offs[i + 1] - q.start;
        q.T = sh.temp[i];
        q.draw = sh.draw[i] != 0;
        return q;
    } else {
        q.start = __ldg(a.seq_offsets + i);
        end = __ldg(a.seq_offsets + i + 1);
        q.T = __ldg(a.temperature + i);
    }
    q.len = end - q.start;
    const bool in_range = q.start >= 0 && end <= a.total && q.len >= 0;
    q.draw = in_range && q.len >= 1 && q.len <= kMaxStride && temperature_ok(q.T) && sh.bad == 0;
    if (q.draw && a.accept_len != nullptr) q.draw = __ldg(a.accept_len + i) == q.len;
    return q;
}

__device__ __forceinline__ int pseq_of_position(const ProposeArgs& a, const PropShared& sh, int r) {
    if (a.num_seqs > kPSeqs) return seq_of_position(a.seq_offsets, a.num_seqs, r);
    int lo = 0, hi = a.num_seqs - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (sh.offs[mid] <= r)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

// The proposal of row r (sequence i, position m = r - start + 1) once every
// chunk partial of the row is published (in global memory, or already in
// sh.part when one CTA reduced the whole row).  Whole CTA.
template <typename Elem>
__device__ void draw_row(const ProposeArgs& a, PropShared& sh, int r, int i, int m, float T, bool in_smem) {
    constexpr int E = sizeof(Elem);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nch = a.nchunks;
    if (!in_smem)
        for (int k = tid; k < nch; k += kPT) sh.part[k] = __ldcg(a.part + static_cast<size_t>(r) * nch + k);
    __syncthreads();
    if (!(T > 0.0f)) {  // greedy: merge the exact chunk argmaxes
        float M = -INFINITY;
        int I = INT_MAX;
        for (int k = tid; k < nch; k += kPT) merge_argmax(M, I, sh.part[k].x, __float_as_int(sh.part[k].y));
        block_merge_arg(sh, M, I);
        if (tid == 0) a.proposals[r] = I;
        return;
    }
    const float c2 = inv_temp_log2e(T);
    if (warp == 0) {
        // Chunk weights in one scale, the target u * total, and its chunk, by
        // lane blocks of consecutive chunks and one warp scan.
        const int ub = (nch + 31) / 32;
        const int k_lo = min(nch, lane * ub), k_hi = min(nch, k_lo + ub);
        float MC = -INFINITY;
        for (int k = k_lo; k < k_hi; ++k) MC = fmaxf(MC, sh.part[k].x);
        MC = warp_max(MC);
        auto wk = [&](int k) -> float {
            const float2 v = sh.part[k];
            return v.x == -INFINITY ? 0.0f : v.y * ex2_approx(v.x - MC);
        };
        float own = 0.0f;
        int lpos = -1;
        for (int k = k_lo; k < k_hi; ++k) {
            const float w = wk(k);
            own += w;
            if (w > 0.0f) lpos = k;
        }
        float incl = own;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        const float u = decision_uniform(a.seed, a.offset, i, m, kTagPropose);
        const float target = u * __shfl_sync(0xffffffffu, incl, 31);
        const unsigned hit = __ballot_sync(0xffffffffu, k_hi > k_lo && incl > target);
        int chosen = -1;
        float tloc = INFINITY;
        if (hit) {
            const int owner = __ffs(hit) - 1;
            if (lane == owner) {
                float cum = incl - own;
                for (int k = k_lo; k < k_hi; ++k) {
                    const float w = wk(k);
                    if (cum + w > target) {
                        chosen = k;
                        tloc = target - cum;
                        break;
                    }
                    cum += w;
                }
                if (chosen < 0) chosen = lpos;  // rounding inside the block
            }
            chosen = __shfl_sync(0xffffffffu, chosen, owner);
            tloc = __shfl_sync(0xffffffffu, tloc, owner);
        }
        if (chosen < 0) {  // rounding left the target past the last weight
            const int lp = warp_max_int(lpos);
            chosen = lp >= 0 ? lp : 0;
            tloc = INFINITY;
        }
        if (lane == 0) {
            sh.sel_chunk = chosen;
            sh.sel_t = tloc;
            sh.sel_mc = MC;
        }
    }
    __syncthreads();
    // Stage the chosen chunk in shared memory, at the same offset from a
    // 16-byte boundary as in global memory.
    const int c = sh.sel_chunk;
    const float tloc = sh.sel_t, MC = sh.sel_mc;
    const int e0 = c * a.chunk;
    const int n = min(a.chunk, a.vocab - e0);
    const char* row = a.rows + static_cast<int64_t>(r) * a.ld_bytes;
    const Span sp = make_span<E>(row, e0, n);
    const uintptr_t base = sp.sb & ~static_cast<uintptr_t>(15);
    const int skew = static_cast<int>(sp.sb - base);  // byte offset of element 0 in the staged copy
    for (int v = tid; v < sp.nvec; v += kPT)
        *reinterpret_cast<uint4*>(sh.chunk + (sp.lo - base) + 16 * v) =
            __ldcg(reinterpret_cast<const uint4*>(sp.lo) + v);
    if (tid < sp.head)
        *reinterpret_cast<Elem*>(sh.chunk + skew + tid * E) = *reinterpret_cast<const Elem*>(sp.sb + tid * E);
    if (tid >= 32 && tid < 32 + sp.tail) {
        const int j = n - sp.tail + (tid - 32);
        *reinterpret_cast<Elem*>(sh.chunk + skew + j * E) = *reinterpret_cast<const Elem*>(sp.sb + static_cast<size_t>(j) * E);
    }
    __syncthreads();
    // In-order scan: thread t owns the consecutive ids [t * seg, (t + 1) * seg).
    const int seg = (n + kPT - 1) / kPT;
    const int b = min(n, tid * seg), e = min(n, b + seg);
    float own = 0.0f;
    int lp = -1;
    for (int j = b; j < e; ++j) {
        const float w = soft_w(raw_elem<Elem>(sh.chunk + skew + j * E), c2, MC);
        own += w;
        if (w > 0.0f) lp = j;
    }
    float incl = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) sh.red_s[warp] = incl;
    __syncthreads();
    float before = 0.0f;
    for (int w = 0; w < warp; ++w) before += sh.red_s[w];
    incl += before;
    // First thread whose running sum passes the target, and the last id with
    // positive weight.
    const bool mine = e > b && incl > tloc;
    const unsigned hw = __ballot_sync(0xffffffffu, mine);
    const int lpw = warp_max_int(lp);
    if (lane == 0) {
        sh.red_i[warp] = hw ? warp * 32 + __ffs(hw) - 1 : INT_MAX;
        sh.red_j[warp] = lpw;
    }
    __syncthreads();
    int owner = INT_MAX, lastp = -1;
    for (int w = 0; w < kPW; ++w) {
        owner = min(owner, sh.red_i[w]);
        lastp = max(lastp, sh.red_j[w]);
    }
    if (owner == INT_MAX) {
        if (tid == 0) a.proposals[r] = e0 + (lastp >= 0 ? lastp : 0);
    } else if (tid == owner) {
        float cum = incl - own;
        int found = -1;
        for (int j = b; j < e; ++j) {
            cum += soft_w(raw_elem<Elem>(sh.chunk + skew + j * E), c2, MC);
            if (cum > tloc) {
                found = j;
                break;
            }
        }
        if (found < 0) found = lp;  // rounding inside this thread's ids
        a.proposals[r] = e0 + found;
    }
}

// One chunk of a row in registers: the thread's 16-byte vectors of the
// aligned interior (-inf past it) and at most one head or tail element.
template <typename Elem>
struct ChunkRegs {
    uint4 v[kPVec];
    float xs;
    int js;    // chunk-relative id of xs, -1 if none
};

template <typename Elem>
__device__ __forceinline__ void load_chunk(const ProposeArgs& a, const char* row, int c, ChunkRegs<Elem>& cr) {
    constexpr int E = sizeof(Elem);
    constexpr uint32_t kNeg = E == 2 ? 0xff80ff80u : 0xff800000u;  // -inf pattern
    const int tid = threadIdx.x;
    const int e0 = c * a.chunk;
    const int n = min(a.chunk, a.vocab - e0);
    const Span sp = make_span<E>(row, e0, n);
#pragma unroll
    for (int k = 0; k < kPVec; ++k) {
        const int vi = tid + k * kPT;
        cr.v[k] = vi < sp.nvec ? __ldcs(reinterpret_cast<const uint4*>(sp.lo) + vi) : make_uint4(kNeg, kNeg, kNeg, kNeg);
    }
    cr.js = -1;
    if (tid < sp.head) cr.js = tid;
    else if (tid >= 32 && tid < 32 + sp.tail) cr.js = n - sp.tail + (tid - 32);
    cr.xs = cr.js >= 0 ? raw_elem<Elem>(reinterpret_cast<const unsigned char*>(sp.sb) + static_cast<size_t>(cr.js) * E)
                       : -INFINITY;
}

// The warp's share of the chunk's softmax partial (mc, s) or exact argmax
// (max, lowest id), stored in sh.wpart[c][warp]; no block barrier, so warps
// run ahead of each other.
template <typename Elem>
__device__ __forceinline__ void reduce_chunk(const ProposeArgs& a, PropShared& sh, const char* row, int c,
                                             const ChunkRegs<Elem>& cr, bool soft, float c2) {
    constexpr int E = sizeof(Elem);
    constexpr int kVec = 16 / E;
    const int tid = threadIdx.x;
    if (soft) {
        float mt = cr.xs;
#pragma unroll
        for (int k = 0; k < kPVec; ++k) mt = fmaxf(mt, vec_max<E>(cr.v[k]));
        float M = -INFINITY, S = 0.0f;
        if (mt != -INFINITY) {
            const float mc = mt * c2;
            const uint64_t C2 = pack_f2(c2, c2), NMC = pack_f2(-mc, -mc);
            uint64_t acc = 0;
#pragma unroll
            for (int k = 0; k < kPVec; ++k) soft_vec<E>(cr.v[k], C2, NMC, acc);
            float s0, s1;
            unpack_f2(acc, s0, s1);
            S = (s0 + s1) + (cr.xs != -INFINITY ? soft_w(cr.xs, c2, mc) : 0.0f);
            M = mc;
        }
        warp_merge_mc2(M, S);
        if ((tid & 31) == 0) sh.wpart[c][tid >> 5] = make_float2(M, S);
        return;
    }
    const int e0 = c * a.chunk;
    const Span sp = make_span<E>(row, e0, min(a.chunk, a.vocab - e0));
    float M = cr.xs;
    int I = cr.js >= 0 ? e0 + cr.js : INT_MAX;
#pragma unroll
    for (int k = 0; k < kPVec; ++k) {
        const int vi = tid + k * kPT;
#pragma unroll
        for (int j = 0; j < kVec; ++j) {
            const float x = vec_elem<E>(cr.v[k], j);
            const int id = e0 + sp.head + vi * kVec + j;
            if (vi < sp.nvec && (x > M || (x == M && id < I))) {
                M = x;
                I = id;
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) merge_argmax(M, I, __shfl_xor_sync(0xffffffffu, M, o), __shfl_xor_sync(0xffffffffu, I, o));
    if ((tid & 31) == 0) sh.wpart[c][tid >> 5] = make_float2(M, __int_as_float(I));
}

template <typename Elem>
__global__ void __launch_bounds__(kPT, kProposeCtasPerSm) propose_kernel(const ProposeArgs a) {
    __shared__ PropShared sh;
    const int tid = threadIdx.x;
    pdl_wait();
    pdl_launch_dependents();
    // Layout: offsets and temperatures of small batches into shared memory;
    // offsets that decrease anywhere make every sequence invalid.
    if (tid == 0) sh.bad = 0;
    __syncthreads();
    bool bad = false;
    const bool small = a.num_seqs <= kPSeqs;
    for (int i = tid; i < a.num_seqs; i += kPT) {
        const int s0 = __ldg(a.seq_offsets + i), s1 = __ldg(a.seq_offsets + i + 1);
        bad = bad || s1 < s0;
        if (small) {
            sh.offs[i] = s0;
            sh.temp[i] = __ldg(a.temperature + i);
            sh.acc[i] = a.accept_len != nullptr ? __ldg(a.accept_len + i) : 0;
            if (i == a.num_seqs - 1) sh.offs[i + 1] = s1;
        }
    }
    if (bad) sh.bad = 1;
    __syncthreads();
    if (small) {
        for (int i = tid; i < a.num_seqs; i += kPT) {
            const int s0 = sh.offs[i], s1 = sh.offs[i + 1], len = s1 - s0;
            bool d = s0 >= 0 && s1 <= a.total && len >= 1 && len <= kMaxStride && temperature_ok(sh.temp[i]) &&
                     sh.bad == 0;
            if (d && a.accept_len != nullptr) d = sh.acc[i] == len;
            sh.draw[i] = d ? 1 : 0;
        }
        __syncthreads();
        // Exclusive prefix of the drawn rows per sequence: thread t sums
        // sequences 2t and 2t + 1, then one scan across the block.
        const int lane = tid & 31, warp = tid >> 5;
        int c0 = 0, c1 = 0;
        if (2 * tid < a.num_seqs && sh.draw[2 * tid]) c0 = sh.offs[2 * tid + 1] - sh.offs[2 * tid];
        if (2 * tid + 1 < a.num_seqs && sh.draw[2 * tid + 1]) c1 = sh.offs[2 * tid + 2] - sh.offs[2 * tid + 1];
        int incl = c0 + c1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        if (lane == 31) sh.wsum[warp] = incl;
        __syncthreads();
        int before = 0;
        for (int w = 0; w < warp; ++w) before += sh.wsum[w];
        const int excl = before + incl - (c0 + c1);
        if (2 * tid < a.num_seqs) sh.pref[2 * tid] = excl;
        if (2 * tid + 1 < a.num_seqs) sh.pref[2 * tid + 1] = excl + c0;
        if (tid == kPT - 1) sh.pref[a.num_seqs] = before + incl;  // every drawn row
        __syncthreads();
    }
    static_assert(2 * kPT >= kPSeqs, "one prefix pass covers every sequence");
    // valid[] and the rows that are not drawn.
    const int gt = blockIdx.x * kPT + tid, gn = gridDim.x * kPT;
    for (int i = gt; i < a.num_seqs; i += gn) a.valid[i] = pseq(a, sh, i).draw ? 1 : 0;
    for (int r = gt; r < a.total; r += gn) {
        const int i = pseq_of_position(a, sh, r);
        const PSeq q = pseq(a, sh, i);
        if (!(q.draw && r >= q.start && r < q.start + q.len)) a.proposals[r] = -1;
    }
    // Pieces: each drawn row is cut into `parts` runs of consecutive chunks,
    // as many as keep every CTA busy (a whole row per CTA once the rows
    // outnumber the CTAs); pieces are dealt round-robin.  Large batches
    // enumerate every row and skip the ones that are not drawn.
    const long long n_rows = small ? sh.pref[a.num_seqs] : a.total;
    const int nch = a.nchunks;
    const int parts = static_cast<int>(max(1LL, min(static_cast<long long>(nch), gridDim.x / max(1LL, n_rows))));
    const long long n_pieces = n_rows * parts;
    for (long long pc = blockIdx.x; pc < n_pieces; pc += gridDim.x) {
        const int j = static_cast<int>(pc / parts);
        const int t = static_cast<int>(pc - static_cast<long long>(j) * parts);
        int i, r;
        if (small) {  // the j-th drawn row: last sequence whose prefix is <= j
            int lo = 0, hi = a.num_seqs - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (sh.pref[mid] <= j)
                    lo = mid;
                else
                    hi = mid - 1;
            }
            i = lo;
            r = sh.offs[i] + (j - sh.pref[i]);
        } else {
            if (tid == 0) {
                const int ii = pseq_of_position(a, sh, j);
                const PSeq q0 = pseq(a, sh, ii);
                sh.item_i = ii;
                sh.item_r = (q0.draw && j >= q0.start && j < q0.start + q0.len) ? j : -1;
            }
            __syncthreads();
            i = sh.item_i;
            r = sh.item_r;
            __syncthreads();
            if (r < 0) continue;  // uniform across the CTA
        }
        const PSeq q = pseq(a, sh, i);
        const bool soft = q.T > 0.0f;
        const float c2 = soft ? inv_temp_log2e(q.T) : 0.0f;
        const char* row = a.rows + static_cast<int64_t>(r) * a.ld_bytes;
        const int c_lo = static_cast<int>(static_cast<long long>(t) * nch / parts);
        const int c_hi = static_cast<int>(static_cast<long long>(t + 1) * nch / parts);
        // Software pipeline: chunk c + 1 is in flight while chunk c is reduced.
        ChunkRegs<Elem> cur, nxt;
        load_chunk<Elem>(a, row, c_lo, cur);
        for (int c = c_lo; c < c_hi; ++c) {
            if (c + 1 < c_hi) load_chunk<Elem>(a, row, c + 1, nxt);
            reduce_chunk<Elem>(a, sh, row, c, cur, soft, c2);
            cur = nxt;
        }
        // Chunk partials from the warps' shares, one thread per chunk.
        __syncthreads();
        for (int c = c_lo + tid; c < c_hi; c += kPT) {
            float2 part;
            if (soft) {
                float M = -INFINITY, S = 0.0f;
                for (int w = 0; w < kPW; ++w) merge_mc(M, S, sh.wpart[c][w].x, sh.wpart[c][w].y);
                part = make_float2(M, S);
            } else {
                float M = -INFINITY;
                int I = INT_MAX;
                for (int w = 0; w < kPW; ++w) merge_argmax(M, I, sh.wpart[c][w].x, __float_as_int(sh.wpart[c][w].y));
                part = make_float2(M, __int_as_float(I));
            }
            sh.part[c] = part;
            if (parts > 1) {
                a.part[static_cast<size_t>(r) * nch + c] = part;
                __threadfence();  // published before the row count below
            }
        }
        __syncthreads();
        if (parts > 1) {  // the CTA that completes the row draws it
            if (tid == 0) {
                __threadfence();
                sh.last = atomicAdd(a.row_count + r, 1) == parts - 1;
            }
            __syncthreads();
            if (sh.last) {
                __threadfence();
                draw_row<Elem>(a, sh, r, i, r - q.start + 1, q.T, false);
                if (tid == 0) a.row_count[r] = 0;  // ready for the next call
            }
        } else {
            draw_row<Elem>(a, sh, r, i, r - q.start + 1, q.T, true);
        }
        __syncthreads();
    }
}

}  // namespace

cudaError_t launch_propose(const ProposeArgs& a, int elem_bytes, int grid, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kPT);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return elem_bytes == 2 ? cudaLaunchKernelEx(&cfg, propose_kernel<__nv_bfloat16>, a)
                           : cudaLaunchKernelEx(&cfg, propose_kernel<float>, a);
}

}  // namespace isd
