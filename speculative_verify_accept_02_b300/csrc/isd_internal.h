// Internal declarations of libisd shared by the host API and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace isd {

// One pipeline stage of the streaming kernel holds one chunk of one row.
constexpr int kStageBytes = 16384;

// Chunking of a vocabulary row: nchunks pieces of `chunk` elements (the last
// may be shorter).  `chunk` is a multiple of the 16-byte vector width and,
// with up to one vector of alignment slack, fits one stage.
struct Chunking {
    int elem_bytes;
    int chunk;
    int nchunks;
};

inline Chunking make_chunking(int vocab, int elem_bytes) {
    const int vec = 16 / elem_bytes;
    const int chunk_max = ((kStageBytes - 16) / elem_bytes) / vec * vec;
    Chunking c;
    c.elem_bytes = elem_bytes;
    c.nchunks = (vocab + chunk_max - 1) / chunk_max;
    if (c.nchunks < 1) c.nchunks = 1;
    const int even = (vocab + c.nchunks - 1) / c.nchunks;
    c.chunk = (even + vec - 1) / vec * vec;
    return c;
}

// Per-(row, chunk) streaming pass: softmax partials (max, sum of exp2) for
// T > 0 rows, (max, lowest argmax id) for T = 0 rows, and the logit of the
// proposed token of each verified row.
struct StatsArgs {
    const char* rows0;          // verify: anchor p; propose: qnew
    int64_t ld0_bytes;
    const char* rows1;          // verify: proposal q; propose: unused
    int64_t ld1_bytes;
    const int32_t* tokens;      // verify: x_k (gathered); propose: null
    const int32_t* seq_offsets;
    const float* temperature;
    const int32_t* accept_len;  // propose: skip sequences with a_i != L_i; else null
    int num_seqs;
    int total;
    int vocab;
    int chunk;
    int nchunks;
    int two_rows;               // 1: verify (slot 2r = p row, 2r+1 = q row); 0: propose
    long long n_items;          // slots * nchunks
    float2* part;               // [slots * nchunks]
    float* zx;                  // [slots] gathered logit (verify)
    int* zero_ptr;              // counters of the following kernel, zeroed here
    int zero_count;
    int* err;                   // error word (bounded waits)
};

struct VerifyFinishArgs {
    const char* p;
    int64_t ldp_bytes;
    const char* q;
    int64_t ldq_bytes;
    const int32_t* tokens;
    const int32_t* seq_offsets;
    const float* temperature;
    int num_seqs;
    int total;
    int vocab;
    int chunk;
    int nchunks;
    uint64_t seed;
    uint64_t offset;
    const float2* part;
    const float* zx;
    float2* tail_part;          // [num_seqs * nchunks]
    int* tail_count;            // [num_seqs]
    const int* err;
    int32_t* accept_len;
    int32_t* out_tokens;
    float* ratio;
    float* alpha;
};

struct ProposeSampleArgs {
    const char* rows;
    int64_t ld_bytes;
    const int32_t* seq_offsets;
    const float* temperature;
    const int32_t* accept_len;
    int num_seqs;
    int total;
    int vocab;
    int chunk;
    int nchunks;
    uint64_t seed;
    uint64_t offset;
    const float2* part;
    const int* err;
    int32_t* proposals;
    uint8_t* valid;
};

// Launchers (return the launch's cudaError_t).
cudaError_t launch_stats(const StatsArgs& a, int elem_bytes, int grid, cudaStream_t stream);
cudaError_t launch_verify_finish(const VerifyFinishArgs& a, int elem_bytes, cudaStream_t stream);
cudaError_t launch_propose_sample(const ProposeSampleArgs& a, int elem_bytes, cudaStream_t stream);
cudaError_t launch_alpha(const float* ratio, const int32_t* seq_offsets, int num_seqs, int total,
                         float* alpha_per_seq, float* alpha_mean, cudaStream_t stream);

// Resident CTAs of the streaming kernel per SM.
constexpr int kStatsCtasPerSm = 2;

}  // namespace isd
