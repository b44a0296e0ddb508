// Internal declarations of libisd shared by the host API and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/isd.h"

namespace isd {

// One pipeline stage of the propose kernel holds one chunk of one row; a
// stage of the verify step's stream kernel holds twice as much.
constexpr int kStageBytes = 16384;
constexpr int kVerifyStageBytes = 32768;

// Chunking of a vocabulary row: nchunks pieces of `chunk` elements (the last
// may be shorter).  `chunk` is a multiple of the 16-byte vector width and,
// with up to one vector of alignment slack, fits one stage of stage_bytes.
struct Chunking {
    int elem_bytes;
    int chunk;
    int nchunks;
};

inline Chunking make_chunking(int vocab, int elem_bytes, int stage_bytes = kStageBytes) {
    const int vec = 16 / elem_bytes;
    const int chunk_max = ((stage_bytes - 16) / elem_bytes) / vec * vec;
    Chunking c;
    c.elem_bytes = elem_bytes;
    c.nchunks = (vocab + chunk_max - 1) / chunk_max;
    if (c.nchunks < 1) c.nchunks = 1;
    const int even = (vocab + c.nchunks - 1) / c.nchunks;
    c.chunk = (even + vec - 1) / vec * vec;
    return c;
}

// The propose kernel: every (qnew row, chunk) of the batch.
struct ProposeArgs {
    const char* rows;
    int64_t ld_bytes;
    const int32_t* seq_offsets;
    const float* temperature;
    const int32_t* accept_len;  // null: every valid sequence is drawn
    int num_seqs;
    int total;
    int vocab;
    int chunk;
    int nchunks;
    uint64_t seed;
    uint64_t offset;
    float2* part;               // [total * nchunks] chunk partials
    int* row_count;             // [total] chunks of each row reduced (zero between calls)
    int32_t* proposals;
    uint8_t* valid;
};

// Most chunks per qnew row the propose kernel supports (vocabularies up to
// 1,047,552 bf16 or 523,776 fp32 ids).
constexpr int kMaxProposeChunks = 128;

// Resident CTAs of the propose kernel per SM.
constexpr int kProposeCtasPerSm = 2;

// ---------------------------------------------------------------------------
// Verify step: stream kernel, then draw kernel
// ---------------------------------------------------------------------------

// Control block (workspace); every call leaves it zero for the next one.
// Each counter has a 128-byte line of its own: hundreds of CTAs poll and
// update them concurrently.
struct VerifyCtl {
    alignas(128) int err;                   // error word (bounded waits)
    alignas(128) unsigned long long grab;   // units handed out by the stream kernel (batches, in sequence order)
    alignas(128) int tail_reserve;          // tail slots reserved by decisions
    alignas(128) unsigned long long claim;  // tail-piece tickets handed to workers
    alignas(128) unsigned long long dclaim; // decision tickets (sequence indices) handed to workers
    alignas(128) int ddone;                 // decisions made (their tail slots reserved)
    alignas(128) int finalized;             // sequences whose outputs are complete
    alignas(128) int draw_tail;             // tails queued for their draw
    alignas(128) int draw_claim;            // queued draws handed to drawing warps
    alignas(128) int exited;                // CTAs of the draw kernel that have finished
};

// Tail modes: what the pieces of a draw after a decision reduce.
enum TailMode : int {
    kTailRes = 1,   // T > 0, rejection: residual max(0, p_j - q_j) over row pair j
    kTailSoft = 2,  // T > 0: softmax draw from one row (bonus from p_{L+1}, or a proposal)
    kTailArg = 3    // T = 0: argmax of one row (a proposal)
};

// Sampler of the draws after a decision.
enum Sampler : int {
    kSamplerIcdf = 0,    // inverse CDF in vocabulary order, one uniform per draw
    kSamplerGumbel = 1   // Gumbel-max, one uniform per vocabulary id and draw
};

// Words of a tail descriptor (each a flagged 64-bit word, flag = slot + 1).
enum TailWord : int {
    kTwPRow = 0,   // the drawn row: p_j, p_{L+1}, or a qnew row
    kTwQRow = 1,   // q_j (residual)
    kTwMeta = 2,   // mode | qnew << 4 | tag << 8 | pos << 16 | draws of the sequence << 24
    kTwC2 = 3,     // log2(e) / T
    kTwNz0 = 4,    // log2 of p_j's normaliser in the exp2 domain
    kTwNz1 = 5,    // the same for q_j
    kTwSeq = 6,    // the sequence
    kTwDest = 7,   // >= 0: out_tokens slot; < 0: proposals slot -1 - dest
    kTailWords = 8
};

struct VerifyArgs {
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
    int ck;            // elements of a main chunk (one stage, one unit)
    int nck;           // chunks per row
    int ps;            // elements of a tail piece
    int np;            // pieces per row
    uint64_t seed;
    uint64_t offset;
    float relax_log2;  // log2(1 + tau) of relaxed acceptance, 0 for strict
    int sampler;       // Sampler of the draws after a decision
    VerifyCtl* ctl;
    int* seq_count;    // [C] chunks of the sequence reduced (stream kernel)
    uint64_t* dready;  // [C] flagged word: every chunk of the sequence is reduced
    int* seq_done;     // [C] draws after the decision finished
    // Tails are queued in the order decisions reserve them: a sequence's
    // correction or bonus draw, and in the fused call one draw per qnew row
    // of a sequence that accepted its whole stride.
    int n_tail;        // capacity: C, or C + total when fused
    uint64_t* tdesc;   // [n_tail][kTailWords] flagged descriptor words
    uint64_t* tpart;   // [n_tail][np][kPieceRecWords] flagged piece records: 4 result words, block weights
    int* tcount;       // [n_tail] pieces finished
    int* dqueue;       // [n_tail] tails whose pieces are all finished, in completion order (slot + 1; 0: not yet)
    float2* part;      // [2 * total][nck] per (row slot, chunk) partials
    // The fused call (isd_verify_propose): the next stride's proposals of the
    // sequences that accept their whole stride, drawn from qnew rows.
    int fused;
    const char* qnew;
    int64_t ldqnew_bytes;
    int32_t* proposals;
    uint8_t* valid;
    int32_t* accept_len;
    int32_t* out_tokens;
    float* ratio;
    float* alpha;
    // Bounds of the waits on other CTAs (global-timer nanoseconds), and a
    // check hook: the decision of sequence `stall_seq` (if >= 0) publishes
    // nothing, so that the waits for it run out (isd_debug.h).
    uint64_t wait_ns;
    int stall_seq;
};

// Bytes of a tail piece per row, and the most pieces per row the verify
// kernel supports (vocabularies up to 524,288 bf16 or 262,144 fp32 ids).
constexpr int kPieceBytes = 4096;
constexpr int kMaxPieces = 256;
// A piece record: four flagged result words, then the flagged weight of each
// 512-byte block of the piece (an even count: records are read in 16-byte
// pairs).
constexpr int kPieceBlocks = kPieceBytes / 512;
constexpr int kPieceRecWords = 4 + kPieceBlocks;
static_assert(kPieceRecWords % 2 == 0, "records of whole 16-byte pairs");

// Resident CTAs of the verify step's stream kernel per SM.
constexpr int kVerifyCtasPerSm = 2;

// SMs the stream kernel leaves with one CTA, where a draw-kernel CTA fits
// beside it from the start.
constexpr int kDrawRoomSms = 16;

cudaError_t launch_verify(const VerifyArgs& a, int elem_bytes, int grid, cudaStream_t stream);

// Default bound of the verify kernel's waits on other CTAs (nanoseconds).
constexpr uint64_t kVerifyWaitNs = 4000000000ull;

// What distinguishes the verify entry points: relaxed acceptance, the
// sampler, the fused proposal draws, and the check hooks of isd_debug.h.
struct VerifyOptions {
    float tau = 0.0f;
    int sampler = kSamplerIcdf;
    bool fused = false;
    const void* qnew = nullptr;
    int64_t ld_qnew = 0;
    int32_t* proposals = nullptr;
    uint8_t* valid = nullptr;
    uint64_t wait_ns = kVerifyWaitNs;
    int stall_seq = -1;
};

// The host-side checks of a verify call, everything but the workspace:
// ISD_OK or the status the call returns (it then launches nothing).
isd_status verify_check(const void* p_logits, int64_t ld_p, const void* q_logits, int64_t ld_q, isd_dtype dtype,
                        int vocab, const int32_t* tokens, const int32_t* seq_offsets, int num_seqs,
                        int total_positions, const float* temperature, int32_t* accept_len, int32_t* out_tokens,
                        float* ratio, float* alpha, const VerifyOptions& o);

// Workspace bytes of a verify call (0 for an invalid shape).
size_t verify_workspace(int num_seqs, int total_positions, int vocab, isd_dtype dtype, bool fused);

// Checks, then one launch of the verify kernel.
isd_status verify_run(const void* p_logits, int64_t ld_p, const void* q_logits, int64_t ld_q, isd_dtype dtype,
                      int vocab, const int32_t* tokens, const int32_t* seq_offsets, int num_seqs,
                      int total_positions, const float* temperature, uint64_t seed, uint64_t offset,
                      int32_t* accept_len, int32_t* out_tokens, float* ratio, float* alpha, const VerifyOptions& o,
                      void* workspace, size_t workspace_bytes, void* stream);

// Launchers (return the launch's cudaError_t).
cudaError_t launch_propose(const ProposeArgs& a, int elem_bytes, int grid, cudaStream_t stream);
cudaError_t launch_alpha(const float* ratio, const int32_t* seq_offsets, int num_seqs, int total,
                         float* alpha_per_seq, float* alpha_mean, cudaStream_t stream);

}  // namespace isd
