// KV-slot commit of the stationary-batch loop ("Introspective Diffusion
// Language Models | Summary", §3.3 I-DLM Serving Stack: KV slots are
// allocated with a batched scatter, and the entries of rejected proposals and
// of mask positions are trimmed; which entries a step keeps and what the next
// step verifies follow §3.2).
//
// One CTA does the whole batch: the work is a few entries per sequence
// (at most 64), so the launch, not bandwidth, sets its time, and a single CTA
// gets the batch-wide prefix sums and the stack order with __syncthreads
// alone, without a grid-wide wait.  Three passes over the sequences, a
// thread per sequence and 256 sequences per tile:
//   1. check every sequence and sum the trimmed and the requested slots;
//      on any error write the status and leave every array as it was;
//   2. push each sequence's trimmed slots at the stack top in (sequence,
//      position) order and clear their table entries;
//   3. hand out the top sum(requested) stack entries as one block, sequence
//      i from its exclusive prefix of the counts onward.
// Every table access stays inside the row because pass 1 refuses a batch
// whose in-flight entries or next allocation run past it; every stack access
// stays inside [0, pool_size) because pass 1 refuses a batch whose pushes
// would overrun the pool or whose requests exceed the stack.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/isd_kv.h"

namespace isd {
namespace {

struct KvArgs {
    int32_t* table;             // [num_seqs, ld]
    int64_t ld;
    int32_t* seq_len;           // [num_seqs]
    int32_t* pend;              // [num_seqs]
    int32_t* alloc;             // [num_seqs]
    int32_t* free_slots;        // [pool_size]
    int32_t* free_top;          // [1]
    int pool_size;
    const int32_t* accept_len;  // [num_seqs]
    int num_seqs;
    int num_masks;
    int32_t* status;            // [1]
};

constexpr int kKvErrState = ISD_KV_ERR_STATE;
constexpr int kKvErrAccept = ISD_KV_ERR_ACCEPT;
constexpr int kKvErrSlot = ISD_KV_ERR_SLOT;
constexpr int kKvErrPool = ISD_KV_ERR_POOL;
constexpr int kKvErrCapacity = ISD_KV_ERR_CAPACITY;

constexpr int kKvThreads = 256;
constexpr int kKvWarps = kKvThreads / 32;

struct KvPlan {
    int kept;       // entries of the forward in flight that stay cached
    int next_pend;  // proposals the next forward verifies
    int status;     // 0 or KV error bits of this sequence
    bool ok;        // state well formed (kept and next_pend are meaningful)
};

// One sequence's outcome.  Checks run in the order of the ABI: first the
// state, then the accept length (either stops the sequence), then the
// trimmed slots and the row capacity.
__device__ KvPlan kv_plan(const KvArgs& a, int i, bool check_slots) {
    KvPlan p{0, 0, 0, false};
    const int len = a.seq_len[i], L = a.pend[i], w = a.alloc[i], M = a.num_masks;
    if (len < 0 || L < 0 || w < 0 || static_cast<long long>(len) + w > a.ld || (w == 0 && L != 0) ||
        (w > 0 && static_cast<long long>(w) != 1LL + L + M)) {
        p.status = kKvErrState;
        return p;
    }
    if (w > 0) {
        const int acc = L > 0 ? a.accept_len[i] : 0;  // a proposal-only step verified nothing
        if (acc < 0 || acc > L) {
            p.status = kKvErrAccept;
            return p;
        }
        p.kept = 1 + acc;                            // x_last, then the accepted prefix
        p.next_pend = (L == 0 || acc == L) ? M : 0;  // the masks' proposals stand
    }
    p.ok = true;
    if (check_slots) {
        const int32_t* row = a.table + static_cast<long long>(i) * a.ld + len;
        for (int j = p.kept; j < w; ++j) {
            const int32_t s = row[j];
            if (s < 0 || s >= a.pool_size) p.status |= kKvErrSlot;
        }
    }
    if (static_cast<long long>(len) + p.kept + 1 + p.next_pend + M > a.ld) p.status |= kKvErrCapacity;
    return p;
}

// Exclusive prefix sum of one value per thread over the CTA; *total gets
// the CTA's sum.  Every thread of the CTA must call it.
__device__ int cta_exclusive_scan(int v, int* warp_sums, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, d);
        if (lane >= d) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int s = lane < kKvWarps ? warp_sums[lane] : 0;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, s, d);
            if (lane >= d) s += y;
        }
        if (lane < kKvWarps) warp_sums[lane] = s;
    }
    __syncthreads();
    const int excl = x - v + (warp > 0 ? warp_sums[warp - 1] : 0);
    *total = warp_sums[kKvWarps - 1];
    __syncthreads();  // warp_sums is reused by the next call
    return excl;
}

__global__ void __launch_bounds__(kKvThreads, 1) kv_commit_kernel(KvArgs a) {
    __shared__ int warp_sums[kKvWarps];
    __shared__ int s_status;
    if (threadIdx.x == 0) s_status = 0;
    __syncthreads();
    const int tiles = (a.num_seqs + kKvThreads - 1) / kKvThreads;

    // Pass 1: checks and totals.
    long long pushed = 0, wanted = 0;
    for (int t = 0; t < tiles; ++t) {
        const int i = t * kKvThreads + static_cast<int>(threadIdx.x);
        int f = 0, n = 0;
        if (i < a.num_seqs) {
            const KvPlan p = kv_plan(a, i, true);
            if (p.status) atomicOr(&s_status, p.status);
            if (p.ok) {
                f = a.alloc[i] - p.kept;
                n = 1 + p.next_pend + a.num_masks;
            }
        }
        int ft, nt;
        cta_exclusive_scan(f, warp_sums, &ft);
        cta_exclusive_scan(n, warp_sums, &nt);
        pushed += ft;
        wanted += nt;
    }
    __syncthreads();
    int status = s_status;
    const long long top = *a.free_top;
    if (status == 0) {
        if (top < 0 || top > a.pool_size || top + pushed > a.pool_size)
            status = kKvErrState;
        else if (top + pushed < wanted)
            status = kKvErrPool;
    }
    if (status != 0) {
        if (threadIdx.x == 0) *a.status = status;
        return;  // uniform across the CTA: every thread computed the same status
    }

    // Pass 2: trim.
    long long carry = 0;
    for (int t = 0; t < tiles; ++t) {
        const int i = t * kKvThreads + static_cast<int>(threadIdx.x);
        KvPlan p{0, 0, 0, false};
        int f = 0;
        if (i < a.num_seqs) {
            p = kv_plan(a, i, false);
            f = a.alloc[i] - p.kept;
        }
        int ft;
        const int ex = cta_exclusive_scan(f, warp_sums, &ft);
        if (i < a.num_seqs) {
            int32_t* row = a.table + static_cast<long long>(i) * a.ld + a.seq_len[i];
            int32_t* dst = a.free_slots + top + carry + ex;
            for (int j = p.kept; j < a.alloc[i]; ++j) {
                *dst++ = row[j];
                row[j] = -1;
            }
        }
        carry += ft;
    }
    __syncthreads();  // the pushes are visible to the block before pass 3 reads the stack

    // Pass 3: batched scatter of the next forward's slots.
    const long long block = top + pushed - wanted;
    carry = 0;
    for (int t = 0; t < tiles; ++t) {
        const int i = t * kKvThreads + static_cast<int>(threadIdx.x);
        KvPlan p{0, 0, 0, false};
        int n = 0;
        if (i < a.num_seqs) {
            p = kv_plan(a, i, false);
            n = 1 + p.next_pend + a.num_masks;
        }
        int nt;
        const int ex = cta_exclusive_scan(n, warp_sums, &nt);
        if (i < a.num_seqs) {
            const int len = a.seq_len[i] + p.kept;
            int32_t* row = a.table + static_cast<long long>(i) * a.ld + len;
            const int32_t* src = a.free_slots + block + carry + ex;
            for (int j = 0; j < n; ++j) row[j] = src[j];
            a.seq_len[i] = len;
            a.pend[i] = p.next_pend;
            a.alloc[i] = n;
        }
        carry += nt;
    }
    if (threadIdx.x == 0) {
        *a.free_top = static_cast<int32_t>(block);
        *a.status = 0;
    }
}

}  // namespace
}  // namespace isd

extern "C" isd_status isd_kv_commit(int32_t* table, int64_t ld, int32_t* seq_len, int32_t* pend,
                                    int32_t* alloc, int32_t* free_slots, int32_t* free_top, int pool_size,
                                    const int32_t* accept_len, int num_seqs, int num_masks, int32_t* status,
                                    void* stream) {
    if (num_seqs < 0 || ld < 1 || pool_size < 0 || num_masks < 0 || num_masks > ISD_MAX_STRIDE - 1)
        return ISD_ERR_INVALID_ARG;
    if (!free_top || !status || (pool_size > 0 && !free_slots)) return ISD_ERR_INVALID_ARG;
    if (num_seqs > 0 && (!table || !seq_len || !pend || !alloc || !accept_len)) return ISD_ERR_INVALID_ARG;
    if (num_seqs > ISD_KV_MAX_SEQS) return ISD_ERR_UNSUPPORTED;
    isd::KvArgs a;
    a.table = table;
    a.ld = ld;
    a.seq_len = seq_len;
    a.pend = pend;
    a.alloc = alloc;
    a.free_slots = free_slots;
    a.free_top = free_top;
    a.pool_size = pool_size;
    a.accept_len = accept_len;
    a.num_seqs = num_seqs;
    a.num_masks = num_masks;
    a.status = status;
    isd::kv_commit_kernel<<<1, isd::kKvThreads, 0, static_cast<cudaStream_t>(stream)>>>(a);
    return cudaGetLastError() == cudaSuccess ? ISD_OK : ISD_ERR_CUDA;
}
