// Host side of libisd: the C ABI of include/isd.h — argument checks,
// workspace layout, kernel launches.  No allocation, no synchronisation.
#include <cuda_runtime.h>

#include <algorithm>
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

// Workspace of isd_verify (stream kernel, then draw kernel):
//   [control block | per-sequence draw counts | per-tail piece counts | draw queue |
//    tail descriptors | tail piece records | per (row slot, chunk) partials]
struct VerifyPlan {
    int ck, nck, ps, np;
};

VerifyPlan verify_plan(int vocab, int esz) {
    VerifyPlan pl;
    const Chunking main = isd::make_chunking(vocab, esz, isd::kVerifyStageBytes);
    pl.ck = main.chunk;
    pl.nck = main.nchunks;
    pl.ps = isd::kPieceBytes / esz;
    pl.np = (vocab + pl.ps - 1) / pl.ps;
    return pl;
}

struct VerifyLayout {
    size_t ctl, seq_count, dready, seq_done, tcount, dqueue, tdesc, tpart, part, bytes;
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
    l.dready = off;
    off = align_up(off + sizeof(uint64_t) * C);
    l.seq_done = off;
    off = align_up(off + sizeof(int) * C);
    l.tcount = off;
    off = align_up(off + sizeof(int) * NT);
    l.dqueue = off;
    off = align_up(off + sizeof(int) * NT);
    l.tdesc = off;
    off = align_up(off + sizeof(uint64_t) * isd::kTailWords * NT);
    l.tpart = off;
    off = align_up(off + sizeof(uint64_t) * isd::kPieceRecWords * NT * static_cast<size_t>(pl.np));  // a record per piece
    l.part = off;
    off = align_up(off + sizeof(float2) * 2 * static_cast<size_t>(total) * pl.nck);
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
    return isd::verify_workspace(num_seqs, total_positions, vocab, dtype, false);
}

size_t isd_verify_propose_workspace_bytes(int num_seqs, int total_positions, int vocab, isd_dtype dtype) {
    return isd::verify_workspace(num_seqs, total_positions, vocab, dtype, true);
}

size_t isd_propose_workspace_bytes(int num_seqs, int total_positions, int vocab, isd_dtype dtype) {
    if (num_seqs < 0 || total_positions < 0 || vocab < 1 || !dtype_ok(dtype)) return 0;
    return propose_layout(total_positions, isd::make_chunking(vocab, elem_bytes_of(dtype))).bytes;
}

}  // extern "C"

namespace isd {

isd_status verify_check(const void* p_logits, int64_t ld_p, const void* q_logits, int64_t ld_q, isd_dtype dtype,
                        int vocab, const int32_t* tokens, const int32_t* seq_offsets, int num_seqs,
                        int total_positions, const float* temperature, int32_t* accept_len, int32_t* out_tokens,
                        float* ratio, float* alpha, const VerifyOptions& o) {
    if (num_seqs < 0 || total_positions < 0 || vocab < 1 || !dtype_ok(dtype)) return ISD_ERR_INVALID_ARG;
    if (!(o.tau >= 0.0f) || !std::isfinite(o.tau)) return ISD_ERR_INVALID_ARG;
    if (o.sampler != kSamplerIcdf && o.sampler != kSamplerGumbel) return ISD_ERR_INVALID_ARG;
    if (num_seqs == 0) return ISD_OK;
    if (!p_logits || !q_logits || !tokens || !seq_offsets || !temperature || !accept_len || !out_tokens ||
        !ratio || !alpha)
        return ISD_ERR_INVALID_ARG;
    if (ld_p < vocab || ld_q < vocab) return ISD_ERR_INVALID_ARG;
    if (o.fused && (!o.qnew || !o.proposals || !o.valid || o.ld_qnew < vocab)) return ISD_ERR_INVALID_ARG;
    if (!aligned16(p_logits) || !aligned16(q_logits) || (o.fused && !aligned16(o.qnew))) return ISD_ERR_UNSUPPORTED;
    if (verify_plan(vocab, elem_bytes_of(dtype)).np > kMaxPieces) return ISD_ERR_UNSUPPORTED;
    return ISD_OK;
}

size_t verify_workspace(int num_seqs, int total_positions, int vocab, isd_dtype dtype, bool fused) {
    if (num_seqs < 0 || total_positions < 0 || vocab < 1 || !dtype_ok(dtype)) return 0;
    return verify_layout(num_seqs, total_positions, verify_plan(vocab, elem_bytes_of(dtype)), fused).bytes;
}

isd_status verify_run(const void* p_logits, int64_t ld_p, const void* q_logits, int64_t ld_q, isd_dtype dtype,
                      int vocab, const int32_t* tokens, const int32_t* seq_offsets, int num_seqs,
                      int total_positions, const float* temperature, uint64_t seed, uint64_t offset,
                      int32_t* accept_len, int32_t* out_tokens, float* ratio, float* alpha, const VerifyOptions& o,
                      void* workspace, size_t workspace_bytes, void* stream) {
    const isd_status chk = verify_check(p_logits, ld_p, q_logits, ld_q, dtype, vocab, tokens, seq_offsets,
                                        num_seqs, total_positions, temperature, accept_len, out_tokens, ratio,
                                        alpha, o);
    if (chk != ISD_OK || num_seqs == 0) return chk;
    if (!workspace) return ISD_ERR_INVALID_ARG;
    const int esz = elem_bytes_of(dtype);
    const VerifyPlan pl = verify_plan(vocab, esz);
    const VerifyLayout lay = verify_layout(num_seqs, total_positions, pl, o.fused);
    if (workspace_bytes < lay.bytes || (reinterpret_cast<uintptr_t>(workspace) % kAlign) != 0)
        return ISD_ERR_WORKSPACE;
    char* ws = static_cast<char*>(workspace);
    VerifyArgs va{};
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
    va.ps = pl.ps;
    va.np = pl.np;
    va.seed = seed;
    va.offset = offset;
    va.relax_log2 = o.tau > 0.0f ? std::log2(1.0f + o.tau) : 0.0f;
    va.sampler = o.sampler;
    va.ctl = reinterpret_cast<VerifyCtl*>(ws + lay.ctl);
    va.seq_count = reinterpret_cast<int*>(ws + lay.seq_count);
    va.dready = reinterpret_cast<uint64_t*>(ws + lay.dready);
    va.seq_done = reinterpret_cast<int*>(ws + lay.seq_done);
    va.n_tail = num_seqs + (o.fused ? total_positions : 0);
    va.tdesc = reinterpret_cast<uint64_t*>(ws + lay.tdesc);
    va.tpart = reinterpret_cast<uint64_t*>(ws + lay.tpart);
    va.tcount = reinterpret_cast<int*>(ws + lay.tcount);
    va.dqueue = reinterpret_cast<int*>(ws + lay.dqueue);
    va.part = reinterpret_cast<float2*>(ws + lay.part);
    va.fused = o.fused ? 1 : 0;
    va.qnew = static_cast<const char*>(o.qnew);
    va.ldqnew_bytes = o.ld_qnew * esz;
    va.proposals = o.proposals;
    va.valid = o.valid;
    va.accept_len = accept_len;
    va.out_tokens = out_tokens;
    va.ratio = ratio;
    va.alpha = alpha;
    va.wait_ns = o.wait_ns;
    va.stall_seq = o.stall_seq;
    // Units: at most one per chunk of every p and q row.
    const long long units = (2LL * total_positions + num_seqs) * pl.nck;
    int grid = 1;
    const isd_status gs = resident_grid(units, kVerifyCtasPerSm, &grid);
    if (gs != ISD_OK) return gs;
    // Some SMs keep room for a draw-kernel CTA beside their one stream CTA,
    // so that decisions and draws of finished sequences run during the stream.
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return ISD_ERR_CUDA;
    grid = std::max(1, std::min(grid, kVerifyCtasPerSm * sms - std::min(kDrawRoomSms, sms / 2)));
    if (launch_verify(va, esz, grid, static_cast<cudaStream_t>(stream)) != cudaSuccess) return ISD_ERR_CUDA;
    return ISD_OK;
}

}  // namespace isd

extern "C" {

isd_status isd_verify(const void* p_logits, int64_t ld_p, const void* q_logits, int64_t ld_q,
                      isd_dtype dtype, int vocab, const int32_t* tokens,
                      const int32_t* seq_offsets, int num_seqs, int total_positions,
                      const float* temperature, uint64_t seed, uint64_t offset,
                      int32_t* accept_len, int32_t* out_tokens, float* ratio, float* alpha,
                      void* workspace, size_t workspace_bytes, void* stream) {
    return isd::verify_run(p_logits, ld_p, q_logits, ld_q, dtype, vocab, tokens, seq_offsets, num_seqs,
                           total_positions, temperature, seed, offset, accept_len, out_tokens, ratio, alpha,
                           isd::VerifyOptions{}, workspace, workspace_bytes, stream);
}

isd_status isd_verify_relaxed(const void* p_logits, int64_t ld_p, const void* q_logits, int64_t ld_q,
                              isd_dtype dtype, int vocab, const int32_t* tokens,
                              const int32_t* seq_offsets, int num_seqs, int total_positions,
                              const float* temperature, uint64_t seed, uint64_t offset, float tau,
                              int32_t* accept_len, int32_t* out_tokens, float* ratio, float* alpha,
                              void* workspace, size_t workspace_bytes, void* stream) {
    isd::VerifyOptions o;
    o.tau = tau;
    return isd::verify_run(p_logits, ld_p, q_logits, ld_q, dtype, vocab, tokens, seq_offsets, num_seqs,
                           total_positions, temperature, seed, offset, accept_len, out_tokens, ratio, alpha, o,
                           workspace, workspace_bytes, stream);
}

static isd_status verify_propose_with(const void* p_logits, int64_t ld_p, const void* q_logits, int64_t ld_q,
                                      isd_dtype dtype, int vocab, const int32_t* tokens,
                                      const int32_t* seq_offsets, int num_seqs, int total_positions,
                                      const float* temperature, uint64_t seed, uint64_t offset, float tau,
                                      int sampler, int32_t* accept_len, int32_t* out_tokens, float* ratio,
                                      float* alpha, const void* qnew_logits, int64_t ld_qnew, int32_t* proposals,
                                      uint8_t* valid, void* workspace, size_t workspace_bytes, void* stream) {
    isd::VerifyOptions o;
    o.tau = tau;
    o.sampler = sampler;
    o.fused = true;
    o.qnew = qnew_logits;
    o.ld_qnew = ld_qnew;
    o.proposals = proposals;
    o.valid = valid;
    return isd::verify_run(p_logits, ld_p, q_logits, ld_q, dtype, vocab, tokens, seq_offsets, num_seqs,
                           total_positions, temperature, seed, offset, accept_len, out_tokens, ratio, alpha, o,
                           workspace, workspace_bytes, stream);
}

isd_status isd_verify_propose(const void* p_logits, int64_t ld_p, const void* q_logits, int64_t ld_q,
                              isd_dtype dtype, int vocab, const int32_t* tokens,
                              const int32_t* seq_offsets, int num_seqs, int total_positions,
                              const float* temperature, uint64_t seed, uint64_t offset, float tau,
                              int32_t* accept_len, int32_t* out_tokens, float* ratio, float* alpha,
                              const void* qnew_logits, int64_t ld_qnew, int32_t* proposals, uint8_t* valid,
                              void* workspace, size_t workspace_bytes, void* stream) {
    return verify_propose_with(p_logits, ld_p, q_logits, ld_q, dtype, vocab, tokens, seq_offsets, num_seqs,
                               total_positions, temperature, seed, offset, tau, isd::kSamplerIcdf, accept_len,
                               out_tokens, ratio, alpha, qnew_logits, ld_qnew, proposals, valid, workspace,
                               workspace_bytes, stream);
}

isd_status isd_verify_propose_gumbel(const void* p_logits, int64_t ld_p, const void* q_logits, int64_t ld_q,
                                     isd_dtype dtype, int vocab, const int32_t* tokens,
                                     const int32_t* seq_offsets, int num_seqs, int total_positions,
                                     const float* temperature, uint64_t seed, uint64_t offset, float tau,
                                     int32_t* accept_len, int32_t* out_tokens, float* ratio, float* alpha,
                                     const void* qnew_logits, int64_t ld_qnew, int32_t* proposals, uint8_t* valid,
                                     void* workspace, size_t workspace_bytes, void* stream) {
    return verify_propose_with(p_logits, ld_p, q_logits, ld_q, dtype, vocab, tokens, seq_offsets, num_seqs,
                               total_positions, temperature, seed, offset, tau, isd::kSamplerGumbel, accept_len,
                               out_tokens, ratio, alpha, qnew_logits, ld_qnew, proposals, valid, workspace,
                               workspace_bytes, stream);
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
