// Host side of libisd: the C ABI of include/isd.h — argument checks,
// workspace layout, kernel launches.  No allocation, no synchronisation.
#include <cuda_runtime.h>

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

// Workspace of isd_verify:
//   [err word | chunk partials of the p and q rows | gathered logits |
//    tail partials | tail counters]
struct VerifyLayout {
    size_t err, part, zx, tail_part, tail_count, bytes;
};

VerifyLayout verify_layout(int num_seqs, int total, const Chunking& ck) {
    VerifyLayout l;
    size_t off = 0;
    l.err = off;
    off = align_up(off + sizeof(int));
    l.part = off;
    off = align_up(off + sizeof(float2) * 2 * static_cast<size_t>(total) * ck.nchunks);
    l.zx = off;
    off = align_up(off + sizeof(float) * 2 * static_cast<size_t>(total));
    l.tail_part = off;
    off = align_up(off + sizeof(float2) * static_cast<size_t>(num_seqs) * ck.nchunks);
    l.tail_count = off;
    off = align_up(off + sizeof(int) * static_cast<size_t>(num_seqs));
    l.bytes = off;
    return l;
}

// Workspace of isd_propose: [err word | chunk partials of the qnew rows]
struct ProposeLayout {
    size_t err, part, bytes;
};

ProposeLayout propose_layout(int total, const Chunking& ck) {
    ProposeLayout l;
    size_t off = 0;
    l.err = off;
    off = align_up(off + sizeof(int));
    l.part = off;
    off = align_up(off + sizeof(float2) * static_cast<size_t>(total) * ck.nchunks);
    l.bytes = off;
    return l;
}

// Streaming grid: resident CTAs of the current device, at most one per item.
isd_status stats_grid(long long n_items, int* grid) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return ISD_ERR_CUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return ISD_ERR_CUDA;
    long long g = static_cast<long long>(sms) * isd::kStatsCtasPerSm;
    if (n_items < g) g = n_items;
    *grid = static_cast<int>(g < 1 ? 1 : g);
    return ISD_OK;
}

}  // namespace

extern "C" {

size_t isd_verify_workspace_bytes(int num_seqs, int total_positions, int vocab, isd_dtype dtype) {
    if (num_seqs < 0 || total_positions < 0 || vocab < 1 || !dtype_ok(dtype)) return 0;
    return verify_layout(num_seqs, total_positions, isd::make_chunking(vocab, elem_bytes_of(dtype))).bytes;
}

size_t isd_propose_workspace_bytes(int num_seqs, int total_positions, int vocab, isd_dtype dtype) {
    if (num_seqs < 0 || total_positions < 0 || vocab < 1 || !dtype_ok(dtype)) return 0;
    return propose_layout(total_positions, isd::make_chunking(vocab, elem_bytes_of(dtype))).bytes;
}

isd_status isd_verify(const void* p_logits, int64_t ld_p, const void* q_logits, int64_t ld_q,
                      isd_dtype dtype, int vocab, const int32_t* tokens,
                      const int32_t* seq_offsets, int num_seqs, int total_positions,
                      const float* temperature, uint64_t seed, uint64_t offset,
                      int32_t* accept_len, int32_t* out_tokens, float* ratio, float* alpha,
                      void* workspace, size_t workspace_bytes, void* stream) {
    if (num_seqs < 0 || total_positions < 0 || vocab < 1 || !dtype_ok(dtype)) return ISD_ERR_INVALID_ARG;
    if (num_seqs == 0) return ISD_OK;
    if (!p_logits || !q_logits || !tokens || !seq_offsets || !temperature || !accept_len ||
        !out_tokens || !ratio || !alpha || !workspace)
        return ISD_ERR_INVALID_ARG;
    if (ld_p < vocab || ld_q < vocab) return ISD_ERR_INVALID_ARG;
    if (!aligned16(p_logits) || !aligned16(q_logits)) return ISD_ERR_UNSUPPORTED;
    const int esz = elem_bytes_of(dtype);
    const Chunking ck = isd::make_chunking(vocab, esz);
    const VerifyLayout lay = verify_layout(num_seqs, total_positions, ck);
    if (workspace_bytes < lay.bytes || (reinterpret_cast<uintptr_t>(workspace) % kAlign) != 0)
        return ISD_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    char* ws = static_cast<char*>(workspace);
    int* err = reinterpret_cast<int*>(ws + lay.err);
    float2* part = reinterpret_cast<float2*>(ws + lay.part);
    float* zx = reinterpret_cast<float*>(ws + lay.zx);
    float2* tail_part = reinterpret_cast<float2*>(ws + lay.tail_part);
    int* tail_count = reinterpret_cast<int*>(ws + lay.tail_count);

    const long long n_items = 2LL * total_positions * ck.nchunks;
    if (n_items > 0) {
        isd::StatsArgs sa{};
        sa.rows0 = static_cast<const char*>(p_logits);
        sa.ld0_bytes = ld_p * esz;
        sa.rows1 = static_cast<const char*>(q_logits);
        sa.ld1_bytes = ld_q * esz;
        sa.tokens = tokens;
        sa.seq_offsets = seq_offsets;
        sa.temperature = temperature;
        sa.accept_len = nullptr;
        sa.num_seqs = num_seqs;
        sa.total = total_positions;
        sa.vocab = vocab;
        sa.chunk = ck.chunk;
        sa.nchunks = ck.nchunks;
        sa.two_rows = 1;
        sa.n_items = n_items;
        sa.part = part;
        sa.zx = zx;
        sa.zero_ptr = tail_count;
        sa.zero_count = num_seqs;
        sa.err = err;
        int grid = 1;
        const isd_status gs = stats_grid(n_items, &grid);
        if (gs != ISD_OK) return gs;
        if (isd::launch_stats(sa, esz, grid, st) != cudaSuccess) return ISD_ERR_CUDA;
    }
    isd::VerifyFinishArgs fa{};
    fa.p = static_cast<const char*>(p_logits);
    fa.ldp_bytes = ld_p * esz;
    fa.q = static_cast<const char*>(q_logits);
    fa.ldq_bytes = ld_q * esz;
    fa.tokens = tokens;
    fa.seq_offsets = seq_offsets;
    fa.temperature = temperature;
    fa.num_seqs = num_seqs;
    fa.total = total_positions;
    fa.vocab = vocab;
    fa.chunk = ck.chunk;
    fa.nchunks = ck.nchunks;
    fa.seed = seed;
    fa.offset = offset;
    fa.part = part;
    fa.zx = zx;
    fa.tail_part = tail_part;
    fa.tail_count = tail_count;
    fa.err = err;
    fa.accept_len = accept_len;
    fa.out_tokens = out_tokens;
    fa.ratio = ratio;
    fa.alpha = alpha;
    if (isd::launch_verify_finish(fa, esz, st) != cudaSuccess) return ISD_ERR_CUDA;
    return ISD_OK;
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
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    char* ws = static_cast<char*>(workspace);
    int* err = reinterpret_cast<int*>(ws + lay.err);
    float2* part = reinterpret_cast<float2*>(ws + lay.part);

    const long long n_items = static_cast<long long>(total_positions) * ck.nchunks;
    if (n_items > 0) {
        isd::StatsArgs sa{};
        sa.rows0 = static_cast<const char*>(qnew_logits);
        sa.ld0_bytes = ld * esz;
        sa.rows1 = nullptr;
        sa.ld1_bytes = 0;
        sa.tokens = nullptr;
        sa.seq_offsets = seq_offsets;
        sa.temperature = temperature;
        sa.accept_len = accept_len_or_null;
        sa.num_seqs = num_seqs;
        sa.total = total_positions;
        sa.vocab = vocab;
        sa.chunk = ck.chunk;
        sa.nchunks = ck.nchunks;
        sa.two_rows = 0;
        sa.n_items = n_items;
        sa.part = part;
        sa.zx = nullptr;
        sa.zero_ptr = nullptr;
        sa.zero_count = 0;
        sa.err = err;
        int grid = 1;
        const isd_status gs = stats_grid(n_items, &grid);
        if (gs != ISD_OK) return gs;
        if (isd::launch_stats(sa, esz, grid, st) != cudaSuccess) return ISD_ERR_CUDA;
    }
    isd::ProposeSampleArgs pa{};
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
    pa.part = part;
    pa.err = err;
    pa.proposals = proposals;
    pa.valid = valid;
    if (isd::launch_propose_sample(pa, esz, st) != cudaSuccess) return ISD_ERR_CUDA;
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
