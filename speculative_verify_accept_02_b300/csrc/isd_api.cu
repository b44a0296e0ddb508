// Host side of libisd: the C ABI of include/isd.h — argument checks,
// workspace layout, kernel launches.  No allocation, no synchronisation.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "../../include/isd.h"
#include "isd_internal.h"

namespace {

using isd::Chunking;

constexpr size_t kAlign = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

int elem_bytes_of(isd_dtype dtype) { return dtype == ISD_DTYPE_BF16 ? 2 : 4; }

bool dtype_ok(int dtype) { return dtype == ISD_DTYPE_BF16 || dtype == ISD_DTYPE_F32; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Workspace of isd_verify (persistent kernel):
//   [control block | per-sequence counters | per-sequence tail state |
//    tail-task queue and flags | per (row slot, segment) partials |
//    per (tail sub-chunk, consumer warp) slice partials]
struct VerifyPlan {
    int ck, nck, spseg, nseg, ckt, nt, tpt, ntask;
};

constexpr int kSubChunksPerSegment = 8;  // one main item: 8 x 16 KB
constexpr int kTailSubChunksPerTask = 2;
constexpr double kL2KeepBytes = 40.0 * (1 << 20);  // of the 126 MB L2

VerifyPlan verify_plan(int vocab, int esz) {
    VerifyPlan pl;
    const Chunking main = isd::make_chunking(vocab, esz);
    pl.ck = main.chunk;
    pl.nck = main.nchunks;
    pl.spseg = kSubChunksPerSegment;
    pl.nseg = (pl.nck + pl.spseg - 1) / pl.spseg;
    // Tail sub-chunks hold one piece of p and one of q: half a stage each.
    const int vec = 16 / esz;
    const int tmax = ((isd::kStageBytes / 2 - 16) / esz) / vec * vec;
    pl.nt = (vocab + tmax - 1) / tmax;
    const int even = (vocab + pl.nt - 1) / pl.nt;
    pl.ckt = (even + vec - 1) / vec * vec;
    pl.tpt = kTailSubChunksPerTask;
    pl.ntask = (pl.nt + pl.tpt - 1) / pl.tpt;
    return pl;
}

struct VerifyLayout {
    size_t ctl, seq_count, seq_pending, tail_count, tails, tasks, task_ready, part, tpart, bytes;
};

// Tails: one per sequence (its correction or bonus), plus one per qnew row
// when the call also draws the next proposals.
VerifyLayout verify_layout(int num_seqs, int total, const VerifyPlan& pl, bool fused) {
    VerifyLayout l;
    const size_t C = static_cast<size_t>(num_seqs);
    const size_t NT = C + (fused ? static_cast<size_t>(total) : 0);
    size_t off = 0;
    l.ctl = off;
    off = align_up(off + sizeof(isd::VerifyCtl));
    l.seq_count = off;
    off = align_up(off + sizeof(int) * C);
    l.seq_pending = off;
    off = align_up(off + sizeof(int) * C);
    l.tail_count = off;
    off = align_up(off + sizeof(int) * NT);
    l.tails = off;
    off = align_up(off + sizeof(isd::SeqTail) * NT);
    l.tasks = off;
    off = align_up(off + 2 * sizeof(int4) * NT * pl.ntask);
    l.task_ready = off;
    off = align_up(off + sizeof(int) * NT * pl.ntask);
    l.part = off;
    off = align_up(off + sizeof(float2) * 2 * static_cast<size_t>(total) * pl.nseg);
    l.tpart = off;
    off = align_up(off + sizeof(float2) * NT * pl.nt * 8);  // 8 consumer-warp slices per tail sub-chunk
    l.bytes = off;
    return l;
}

// Workspace of isd_propose: [per-row chunk counters | chunk partials of the qnew rows]
struct ProposeLayout {
    size_t row_count, part, bytes;
};

ProposeLayout propose_layout(int total, const Chunking& ck) {
    ProposeLayout l;
    size_t off = 0;
    l.row_count = off;
    off = align_up(off + sizeof(int) * static_cast<size_t>(total));
    l.part = off;
    off = align_up(off + sizeof(float2) * static_cast<size_t>(total) * ck.nchunks);
    l.bytes = off;
    return l;
}

// Persistent grid: resident CTAs of the current device, at most one per item.
isd_status resident_grid(long long n_items, int ctas_per_sm, int* grid) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return ISD_ERR_CUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return ISD_ERR_CUDA;
    long long g = static_cast<long long>(sms) * ctas_per_sm;
    if (n_items < g) g = n_items;
    *grid = static_cast<int>(g < 1 ? 1 : g);
    return ISD_OK;
}


}  // namespace

extern "C" {

size_t isd_verify_workspace_bytes(int num_seqs, int total_positions, int vocab, isd_dtype dtype) {
    if (num_seqs < 0 || total_positions < 0 || vocab < 1 || !dtype_ok(dtype)) return 0;
    return verify_layout(num_seqs, total_positions, verify_plan(vocab, elem_bytes_of(dtype)), false).bytes;
}

size_t isd_verify_propose_workspace_bytes(int num_seqs, int total_positions, int vocab, isd_dtype dtype) {
    if (num_seqs < 0 || total_positions < 0 || vocab < 1 || !dtype_ok(dtype)) return 0;
    return verify_layout(num_seqs, total_positions, verify_plan(vocab, elem_bytes_of(dtype)), true).bytes;
}

size_t isd_propose_workspace_bytes(int num_seqs, int total_positions, int vocab, isd_dtype dtype) {
    if (num_seqs < 0 || total_positions < 0 || vocab < 1 || !dtype_ok(dtype)) return 0;
    return propose_layout(total_positions, isd::make_chunking(vocab, elem_bytes_of(dtype))).bytes;
}

}  // extern "C"

namespace {

isd_status verify_impl(const void* p_logits, int64_t ld_p, const void* q_logits, int64_t ld_q,
                       isd_dtype dtype, int vocab, const int32_t* tokens,
                       const int32_t* seq_offsets, int num_seqs, int total_positions,
                       const float* temperature, uint64_t seed, uint64_t offset, float tau,
                       int32_t* accept_len, int32_t* out_tokens, float* ratio, float* alpha,
                       bool fused, const void* qnew_logits, int64_t ld_qnew, int32_t* proposals,
                       uint8_t* valid, void* workspace, size_t workspace_bytes, void* stream) {
    if (num_seqs < 0 || total_positions < 0 || vocab < 1 || !dtype_ok(dtype)) return ISD_ERR_INVALID_ARG;
    if (!(tau >= 0.0f) || !std::isfinite(tau)) return ISD_ERR_INVALID_ARG;
    if (num_seqs == 0) return ISD_OK;
    if (!p_logits || !q_logits || !tokens || !seq_offsets || !temperature || !accept_len ||
        !out_tokens || !ratio || !alpha || !workspace)
        return ISD_ERR_INVALID_ARG;
    if (ld_p < vocab || ld_q < vocab) return ISD_ERR_INVALID_ARG;
    if (fused && (!qnew_logits || !proposals || !valid || ld_qnew < vocab)) return ISD_ERR_INVALID_ARG;
    if (!aligned16(p_logits) || !aligned16(q_logits) || (fused && !aligned16(qnew_logits)))
        return ISD_ERR_UNSUPPORTED;
    const int esz = elem_bytes_of(dtype);
    const VerifyPlan pl = verify_plan(vocab, esz);
    if (pl.nt > isd::kMaxTailChunks) return ISD_ERR_UNSUPPORTED;
    const VerifyLayout lay = verify_layout(num_seqs, total_positions, pl, fused);
    if (workspace_bytes < lay.bytes || (reinterpret_cast<uintptr_t>(workspace) % kAlign) != 0)
        return ISD_ERR_WORKSPACE;
    char* ws = static_cast<char*>(workspace);
    isd::VerifyArgs va{};
    va.p = static_cast<const char*>(p_logits);
    va.ldp_bytes = ld_p * esz;
    va.q = static_cast<const char*>(q_logits);
    va.ldq_bytes = ld_q * esz;
    va.tokens = tokens;
    va.seq_offsets = seq_offsets;
    va.temperature = temperature;
    va.num_seqs = num_seqs;
    va.total = total_positions;
    va.vocab = vocab;
    va.ck = pl.ck;
    va.nck = pl.nck;
    va.spseg = pl.spseg;
    va.nseg = pl.nseg;
    va.ckt = pl.ckt;
    va.nt = pl.nt;
    va.tpt = pl.tpt;
    va.ntask = pl.ntask;
    va.n_main = 2LL * total_positions * pl.nseg;
    // Rows of the first position of every sequence, both p and q, kept in L2
    // while they fit in about a third of it.
    va.keep_first = 2.0 * num_seqs * vocab * esz <= kL2KeepBytes ? 1 : 0;
    va.seed = seed;
    va.relax_log2 = tau > 0.0f ? std::log2(1.0f + tau) : 0.0f;
    va.offset = offset;
    va.ctl = reinterpret_cast<isd::VerifyCtl*>(ws + lay.ctl);
    va.seq_count = reinterpret_cast<int*>(ws + lay.seq_count);
    va.seq_pending = reinterpret_cast<int*>(ws + lay.seq_pending);
    va.n_tail = num_seqs + (fused ? total_positions : 0);
    va.fused = fused ? 1 : 0;
    va.qnew = static_cast<const char*>(qnew_logits);
    va.ldqnew_bytes = ld_qnew * esz;
    va.proposals = proposals;
    va.valid = valid;
    va.tail_count = reinterpret_cast<int*>(ws + lay.tail_count);
    va.tails = reinterpret_cast<isd::SeqTail*>(ws + lay.tails);
    va.tasks = reinterpret_cast<int4*>(ws + lay.tasks);
    va.task_ready = reinterpret_cast<int*>(ws + lay.task_ready);
    va.part = reinterpret_cast<float2*>(ws + lay.part);
    va.tpart = reinterpret_cast<float2*>(ws + lay.tpart);
    va.accept_len = accept_len;
    va.out_tokens = out_tokens;
    va.ratio = ratio;
    va.alpha = alpha;
    int grid = 1;
    const isd_status gs = resident_grid(va.n_main, isd::kVerifyCtasPerSm, &grid);
    if (gs != ISD_OK) return gs;
    if (isd::launch_verify(va, esz, grid, static_cast<cudaStream_t>(stream)) != cudaSuccess) return ISD_ERR_CUDA;
    return ISD_OK;
}

}  // namespace

extern "C" {

isd_status isd_verify(const void* p_logits, int64_t ld_p, const void* q_logits, int64_t ld_q,
                      isd_dtype dtype, int vocab, const int32_t* tokens,
                      const int32_t* seq_offsets, int num_seqs, int total_positions,
                      const float* temperature, uint64_t seed, uint64_t offset,
                      int32_t* accept_len, int32_t* out_tokens, float* ratio, float* alpha,
                      void* workspace, size_t workspace_bytes, void* stream) {
    return verify_impl(p_logits, ld_p, q_logits, ld_q, dtype, vocab, tokens, seq_offsets, num_seqs,
                       total_positions, temperature, seed, offset, 0.0f, accept_len, out_tokens, ratio, alpha,
                       false, nullptr, 0, nullptr, nullptr, workspace, workspace_bytes, stream);
}

isd_status isd_verify_relaxed(const void* p_logits, int64_t ld_p, const void* q_logits, int64_t ld_q,
                              isd_dtype dtype, int vocab, const int32_t* tokens,
                              const int32_t* seq_offsets, int num_seqs, int total_positions,
                              const float* temperature, uint64_t seed, uint64_t offset, float tau,
                              int32_t* accept_len, int32_t* out_tokens, float* ratio, float* alpha,
                              void* workspace, size_t workspace_bytes, void* stream) {
    return verify_impl(p_logits, ld_p, q_logits, ld_q, dtype, vocab, tokens, seq_offsets, num_seqs,
                       total_positions, temperature, seed, offset, tau, accept_len, out_tokens, ratio, alpha,
                       false, nullptr, 0, nullptr, nullptr, workspace, workspace_bytes, stream);
}

isd_status isd_verify_propose(const void* p_logits, int64_t ld_p, const void* q_logits, int64_t ld_q,
                              isd_dtype dtype, int vocab, const int32_t* tokens,
                              const int32_t* seq_offsets, int num_seqs, int total_positions,
                              const float* temperature, uint64_t seed, uint64_t offset, float tau,
                              int32_t* accept_len, int32_t* out_tokens, float* ratio, float* alpha,
                              const void* qnew_logits, int64_t ld_qnew, int32_t* proposals, uint8_t* valid,
                              void* workspace, size_t workspace_bytes, void* stream) {
    return verify_impl(p_logits, ld_p, q_logits, ld_q, dtype, vocab, tokens, seq_offsets, num_seqs,
                       total_positions, temperature, seed, offset, tau, accept_len, out_tokens, ratio, alpha,
                       true, qnew_logits, ld_qnew, proposals, valid, workspace, workspace_bytes, stream);
}

isd_status isd_propose(const void* qnew_logits, int64_t ld, isd_dtype dtype, int vocab,
                       const int32_t* seq_offsets, int num_seqs, int total_positions,
                       const float* temperature, uint64_t seed, uint64_t offset,
                       const int32_t* accept_len_or_null, int32_t* proposals, uint8_t* valid,
                       void* workspace, size_t workspace_bytes, void* stream) {
    if (num_seqs < 0 || total_positions < 0 || vocab < 1 || !dtype_ok(dtype)) return ISD_ERR_INVALID_ARG;
    if (num_seqs == 0) return ISD_OK;
    if (!qnew_logits || !seq_offsets || !temperature || !proposals || !valid || !workspace)
        return ISD_ERR_INVALID_ARG;
    if (ld < vocab) return ISD_ERR_INVALID_ARG;
    if (!aligned16(qnew_logits)) return ISD_ERR_UNSUPPORTED;
    const int esz = elem_bytes_of(dtype);
    const Chunking ck = isd::make_chunking(vocab, esz);
    const ProposeLayout lay = propose_layout(total_positions, ck);
    if (workspace_bytes < lay.bytes || (reinterpret_cast<uintptr_t>(workspace) % kAlign) != 0)
        return ISD_ERR_WORKSPACE;
    if (ck.nchunks > isd::kMaxProposeChunks) return ISD_ERR_UNSUPPORTED;
    char* ws = static_cast<char*>(workspace);
    isd::ProposeArgs pa{};
    pa.rows = static_cast<const char*>(qnew_logits);
    pa.ld_bytes = ld * esz;
    pa.seq_offsets = seq_offsets;
    pa.temperature = temperature;
    pa.accept_len = accept_len_or_null;
    pa.num_seqs = num_seqs;
    pa.total = total_positions;
    pa.vocab = vocab;
    pa.chunk = ck.chunk;
    pa.nchunks = ck.nchunks;
    pa.seed = seed;
    pa.offset = offset;
    pa.part = reinterpret_cast<float2*>(ws + lay.part);
    pa.row_count = reinterpret_cast<int*>(ws + lay.row_count);
    pa.proposals = proposals;
    pa.valid = valid;
    int grid = 1;
    const long long n_items = static_cast<long long>(total_positions) * ck.nchunks;
    const isd_status gs = resident_grid(n_items > num_seqs ? n_items : num_seqs, isd::kProposeCtasPerSm, &grid);
    if (gs != ISD_OK) return gs;
    if (isd::launch_propose(pa, esz, grid, static_cast<cudaStream_t>(stream)) != cudaSuccess) return ISD_ERR_CUDA;
    return ISD_OK;
}

isd_status isd_alpha(const float* ratio, const int32_t* seq_offsets, int num_seqs,
                     int total_positions, float* alpha_per_seq, float* alpha_mean, void* stream) {
    if (num_seqs < 0 || total_positions < 0) return ISD_ERR_INVALID_ARG;
    if (num_seqs == 0) return ISD_OK;
    if (!ratio || !seq_offsets || !alpha_per_seq || !alpha_mean) return ISD_ERR_INVALID_ARG;
    if (isd::launch_alpha(ratio, seq_offsets, num_seqs, total_positions, alpha_per_seq, alpha_mean,
                          static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return ISD_ERR_CUDA;
    return ISD_OK;
}

const char* isd_status_string(isd_status status) {
    switch (status) {
        case ISD_OK: return "ok";
        case ISD_ERR_INVALID_ARG: return "invalid argument";
        case ISD_ERR_UNSUPPORTED: return "unsupported layout (logits must be 16-byte aligned)";
        case ISD_ERR_WORKSPACE: return "workspace too small or misaligned";
        case ISD_ERR_CUDA: return "CUDA error";
    }
    return "unknown status";
}

}  // extern "C"
