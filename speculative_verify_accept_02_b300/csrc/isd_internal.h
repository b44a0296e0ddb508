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
// Persistent verify kernel
// ---------------------------------------------------------------------------

// Control block (workspace); every call leaves it zero for the next one.
// Each counter has a 128-byte line of its own: hundreds of CTAs poll and
// update them concurrently.
struct VerifyCtl {
    alignas(128) int err;                  // error word (bounded waits)
    alignas(128) unsigned long long grab;  // main items handed out (dynamic scheduling)
    alignas(128) int tail_reserve;         // tail-task slots reserved by decisions
    alignas(128) int tail_claim;           // tail-task tickets handed to producers
    alignas(128) int finalized;            // sequences whose outputs are complete
    alignas(128) int exited;               // CTAs that have finished
};

// Tail kinds: which row(s) the work after a decision reads.
enum TailMode : int {
    kTailRes = 2,   // T > 0, rejection: residual max(0, p_j - q_j) over row pair j
    kTailSoft = 3,  // T > 0: softmax draw from one row (bonus from p_{L+1}, or a proposal)
    kTailArg = 4    // T = 0: argmax of one row (a proposal)
};
// Flag on a tail mode: its row is a qnew row (a proposal draw of the fused
// verify-and-propose call), not a p row.
constexpr int kTailQnew = 8;

// What a sequence's tail needs, written by its decision (48 bytes).
// What a tail (one draw after a decision) needs: written by the decision,
// read by the tail's producers and its selection (48 bytes).
struct alignas(16) SeqTail {
    int mode;         // TailMode, with kTailQnew for a proposal row
    int a;            // accept length of the sequence
    int prow, qrow;   // rows: p_j (or p_{L+1}, or the qnew row) and q_j
    float c2;         // log2(e) / T
    float nz0;        // p_j: log2 of its normaliser, p_j(v) = exp2(x_v c2 - nz0)
    float nz1;        // q_j: the same
    int seq;          // the sequence
    int pos;          // position of the draw's uniform (1-based)
    int tag;          // the uniform's purpose (CORRECT, BONUS or PROPOSE)
    int dest;         // >= 0: out_tokens slot; < 0: proposals slot -1 - dest
    int pad;
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
    int ck;           // elements of a main sub-chunk (one stage)
    int nck;          // main sub-chunks per row
    int spseg;        // sub-chunks per segment (one main item)
    int nseg;         // segments per row
    int ckt;          // elements of a tail sub-chunk (half a stage per row)
    int nt;           // tail sub-chunks per row
    int tpt;          // tail sub-chunks per tail task
    int ntask;        // tail tasks per sequence
    long long n_main; // 2 * total * nseg main items
    int keep_first;   // 1: first-position rows of T > 0 sequences are kept in L2 for their tails
    uint64_t seed;
    uint64_t offset;
    float relax_log2; // log2(1 + tau) of relaxed acceptance, 0 for strict
    VerifyCtl* ctl;
    int* seq_count;   // [C] main items finished
    // Tails are indexed by tail id: sequence i's correction or bonus is tail
    // i; with `fused`, the proposal draw of qnew row r is tail C + r.
    int n_tail;       // C, or C + total when fused
    int* tail_count;  // [n_tail] tail tasks finished
    SeqTail* tails;   // [n_tail]
    int4* tasks;      // [n_tail * ntask][2] task records in reservation order:
                      // {tail id, task, mode, row}, {q row, c2, nz0, nz1}
    int* task_ready;  // [n_tail * ntask] 1 once the slot's task is published
    float2* part;     // [2 * total * nseg] per (row slot, segment) partials
    float2* tpart;    // [n_tail * nt * 8] per (tail sub-chunk, consumer warp) slice partials
    int* seq_pending; // [C] draws of the sequence still to finish
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
};

// Largest number of tail sub-chunks per row the verify kernel supports
// (vocabularies up to 523,264 bf16 or 261,632 fp32 ids).
constexpr int kMaxTailChunks = 128;

// Resident CTAs of the verify kernel per SM.
constexpr int kVerifyCtasPerSm = 2;

cudaError_t launch_verify(const VerifyArgs& a, int elem_bytes, int grid, cudaStream_t stream);

// Launchers (return the launch's cudaError_t).
cudaError_t launch_propose(const ProposeArgs& a, int elem_bytes, int grid, cudaStream_t stream);
cudaError_t launch_alpha(const float* ratio, const int32_t* seq_offsets, int num_seqs, int total,
                         float* alpha_per_seq, float* alpha_mean, cudaStream_t stream);

}  // namespace isd
