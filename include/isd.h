/*
 * isd.h — C ABI of libisd, the per-step verify-and-propose pass of
 * Introspective Strided Decoding (ISD) over vocabulary logits, for one
 * NVIDIA B300 (sm_103a).
 *
 * The method is from "Introspective Diffusion Language Models | Summary":
 *   §2 Background and Motivation   — introspective acceptance rate alpha;
 *   §3.2 Introspective Strided Decoding — strict acceptance with probability
 *        min(1, p_k(x_k)/q_k(x_k)), correction from normalize(max(0, p - q))
 *        at the first rejection, bonus token from the final causal anchor,
 *        proposal-only step after a rejection;
 *   §3.3 I-DLM Serving Stack — argmax proposals with strict verification
 *        (greedy, temperature 0); the verification runs as fused kernels;
 *   §3.1 Introspective-Consistency Training — next-token logit shift.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Memory.   Every pointer argument is a DEVICE pointer owned by the caller
 *           (logits, offsets, temperatures, outputs, workspace).  The library
 *           allocates nothing, never synchronises, keeps no state of its own
 *           between calls, and enqueues its kernels on `stream` (a
 *           cudaStream_t; NULL means the legacy default stream).  Results are
 *           valid once the stream reaches them.
 * Batch.    num_seqs = C sequences.  seq_offsets[C+1] is the exclusive prefix
 *           sum of the per-sequence strides L_i (the number of proposals of
 *           sequence i), non-decreasing, seq_offsets[0] = 0 and
 *           seq_offsets[C] = total_positions = sum_i L_i.  Sequence i owns
 *           positions seq_offsets[i] .. seq_offsets[i+1]-1.
 * Rows.     Logits are row-major [rows, ld] in bf16 or fp32; only the first
 *           `vocab` entries of a row are read; ld >= vocab (elements).  The
 *           base pointer must be 16-byte aligned (ISD_ERR_UNSUPPORTED
 *           otherwise); ld is free.  Logits must not be NaN or +inf; -inf is
 *           allowed, but every row needs a finite entry.
 *   p (anchor, next-token shifted, §3.1): L_i + 1 rows per sequence; row
 *           seq_offsets[i] + i + (k-1) holds p_k, the logits that score x_k
 *           (k <= L_i); row seq_offsets[i] + i + L_i is the final anchor.
 *   q (proposal): L_i rows per sequence; row seq_offsets[i] + (k-1) holds
 *           q_k, the logits that produced x_k.
 * Temperature.  temperature[i] = T_i >= 0 applies to p and q alike (logits
 *           divided by T_i).  T_i = 0 is greedy: a proposal is accepted iff
 *           it is the argmax of p_k (lowest id on ties), the correction and
 *           the bonus are argmaxes, and q is not read.
 * Random numbers.  Each decision draws one uniform u in [0, 1) from
 *           Philox4x64-10 (Salmon et al., SC'11) with key (seed, 0) and
 *           counter (offset, i, k, tag), tag ACCEPT=0 / CORRECT=1 / BONUS=2 /
 *           PROPOSE=3; u is the top 24 bits of output word 0 times 2^-24.
 *           The caller advances `offset` once per decode step; verify and
 *           propose may share an offset (their tags differ).  Sampling is by
 *           inverse CDF in vocabulary order: the smallest id whose running
 *           weight exceeds u times the total weight.
 * Validity. A sequence whose stride is outside [1, 32], whose temperature is
 *           negative, subnormal or not finite, whose range lies outside
 *           [0, total_positions], or (verify) whose tokens lie outside
 *           [0, vocab) is invalid: it is not computed, accept_len[i] = -1,
 *           its output slots are -1 and its ratios and alpha NaN.  Invalid
 *           sequences never trap the device.
 * Workspace.  Caller-owned device memory of at least the size the matching
 *           *_workspace_bytes() reports, 256-byte aligned, ZERO-FILLED
 *           before its first use; every call leaves it reusable for the next
 *           call of the same entry point.  Calls that share a workspace must
 *           be ordered (same stream or events).  isd_verify's internal
 *           waits are bounded: if one ever gives up (a hardware fault, not an
 *           input error), every accept_len reads -2 and the workspace must be
 *           zero-filled again.  isd_propose has no internal waits.
 * Errors.   Host-side checks return a status and launch nothing.  A CUDA
 *           launch error returns ISD_ERR_CUDA (the sticky error is left for
 *           the caller to inspect).
 */
#ifndef ISD_H_
#define ISD_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define ISD_API __attribute__((visibility("default")))
#else
#define ISD_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ISD_OK = 0,
    ISD_ERR_INVALID_ARG = 1,   /* null pointer, negative size, ld < vocab, bad dtype */
    ISD_ERR_UNSUPPORTED = 2,   /* logits base not 16-byte aligned; isd_verify: vocab above
                                  524,288 (bf16) or 262,144 (fp32); isd_propose: vocab above
                                  1,047,552 (bf16) or 523,776 (fp32) */
    ISD_ERR_WORKSPACE = 3,     /* workspace too small or not 256-byte aligned */
    ISD_ERR_CUDA = 4           /* a CUDA call failed (launch or device query) */
} isd_status;

typedef enum { ISD_DTYPE_BF16 = 0, ISD_DTYPE_F32 = 1 } isd_dtype;

/* Largest stride L_i one sequence may verify (one warp ballot). */
#define ISD_MAX_STRIDE 32

/* Bytes of workspace isd_verify needs for this batch shape. */
ISD_API size_t isd_verify_workspace_bytes(int num_seqs, int total_positions, int vocab, isd_dtype dtype);

/*
 * isd_verify — verify the previous stride's proposals of every sequence and
 * emit the accepted prefix plus one token (§2, §3.2, §3.3).
 *
 * Per sequence i (L = L_i, T = T_i):
 *   ratio_k  = min(1, p_k(x_k) / q_k(x_k)), p_k = softmax(P_k / T),
 *              q_k = softmax(Q_k / T)   (T = 0: 1 if x_k is argmax P_k else 0)
 *   alpha_i  = (1/L) sum_{k=1..L} ratio_k          (all L positions, §2)
 *   a_i      = number of leading k with u_k < ratio_k (T = 0: ratio_k = 1),
 *              u_k the ACCEPT uniform of position k
 *   token    = a_i < L: draw from normalize(max(0, p_j - q_j)), j = a_i + 1,
 *                       with the CORRECT uniform of position j (all-zero
 *                       residual: from p_j); T = 0: argmax P_j
 *              a_i = L: draw from p_{L+1} with the BONUS uniform of position
 *                       L + 1; T = 0: argmax P_{L+1}
 *
 * p_logits   [total + C, ld_p] anchor logits (layout above), bf16 or fp32
 * q_logits   [total, ld_q]     proposal logits, same dtype as p
 * tokens     [total] int32     x_k, the previously proposed tokens
 * seq_offsets[C + 1] int32, temperature [C] float32 (see conventions)
 * seed, offset               Philox key word and step counter
 * accept_len [C] int32 out    a_i (-1 invalid sequence, -2 internal timeout)
 * out_tokens [total + C] out  L_i + 1 slots per sequence starting at
 *                             seq_offsets[i] + i: x_1..x_{a_i}, then the
 *                             correction or bonus token, then -1
 * ratio      [total] float out ratio_k per position (NaN if invalid)
 * alpha      [C] float out     alpha_i (NaN if invalid)
 * workspace, workspace_bytes  scratch (see conventions)
 */
ISD_API isd_status isd_verify(const void* p_logits, int64_t ld_p, const void* q_logits, int64_t ld_q,
                              isd_dtype dtype, int vocab, const int32_t* tokens,
                              const int32_t* seq_offsets, int num_seqs, int total_positions,
                              const float* temperature, uint64_t seed, uint64_t offset,
                              int32_t* accept_len, int32_t* out_tokens, float* ratio, float* alpha,
                              void* workspace, size_t workspace_bytes, void* stream);

/*
 * isd_verify_relaxed — isd_verify with the relaxed acceptance of the pages'
 * ablation (experiments, Table 4: the acceptance ratio multiplied by 1 + tau).
 * Each accept test becomes u_k < min(1, (1 + tau) p_k(x_k) / q_k(x_k)); the
 * correction is still drawn from normalize(max(0, p_j - q_j)), and ratio and
 * alpha still report the strict min(1, p_k(x_k)/q_k(x_k)).  Relaxation gives
 * up exact preservation of the anchor distribution.  tau = 0 is isd_verify;
 * T = 0 (greedy) is unaffected.  tau must be finite and >= 0
 * (ISD_ERR_INVALID_ARG otherwise).  Every other argument as isd_verify; the
 * two share a workspace size.
 */
ISD_API isd_status isd_verify_relaxed(const void* p_logits, int64_t ld_p, const void* q_logits, int64_t ld_q,
                                      isd_dtype dtype, int vocab, const int32_t* tokens,
                                      const int32_t* seq_offsets, int num_seqs, int total_positions,
                                      const float* temperature, uint64_t seed, uint64_t offset, float tau,
                                      int32_t* accept_len, int32_t* out_tokens, float* ratio, float* alpha,
                                      void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of workspace isd_verify_propose needs for this batch shape. */
ISD_API size_t isd_verify_propose_workspace_bytes(int num_seqs, int total_positions, int vocab, isd_dtype dtype);

/*
 * isd_verify_propose — one call that does isd_verify_relaxed (tau = 0:
 * isd_verify) and then isd_propose with this call's accept lengths: the
 * fused step of Summary §3.2, where one forward verifies the pending
 * proposals and its mask positions propose the next stride.  Proposals are
 * drawn only for sequences that accept their whole stride (valid[i] = 1);
 * the others get valid[i] = 0 and proposals -1, as isd_propose with
 * accept_len_or_null does.  Every output equals that of the two separate
 * calls on the same arguments (same uniforms); the proposal draws run in the
 * verify call's draw kernel, right after the decision that keeps them.
 *
 * Arguments: those of isd_verify_relaxed, then
 * qnew_logits, ld_qnew  [total, ld_qnew] this forward's mask-position logits
 *                       (layout of q), same dtype as p, 16-byte aligned base
 * proposals [total] int32 out, valid [C] uint8 out
 * workspace of at least isd_verify_propose_workspace_bytes() (the rules of
 * every workspace), not shared with isd_verify calls in flight.
 */
ISD_API isd_status isd_verify_propose(const void* p_logits, int64_t ld_p, const void* q_logits, int64_t ld_q,
                                      isd_dtype dtype, int vocab, const int32_t* tokens,
                                      const int32_t* seq_offsets, int num_seqs, int total_positions,
                                      const float* temperature, uint64_t seed, uint64_t offset, float tau,
                                      int32_t* accept_len, int32_t* out_tokens, float* ratio, float* alpha,
                                      const void* qnew_logits, int64_t ld_qnew, int32_t* proposals,
                                      uint8_t* valid, void* workspace, size_t workspace_bytes, void* stream);

/*
 * isd_verify_propose_gumbel — isd_verify_propose with Gumbel-max draws in
 * place of inverse-CDF draws for the correction, the bonus token and the
 * proposals: the sampler of the pages' fused verification kernel (§3.3,
 * "online softmax and Gumbel-max correction").  A draw from weights w gives
 * the id that maximises log w_v - log(-log u_v) over the ids with w_v > 0,
 * the lower id on ties, with one uniform per vocabulary id and draw: u_v
 * from Philox4x64-10 with key (seed, 0) and counter (offset, i, position,
 * 16 + tag + 256 floor(v / 4)), output word v mod 4, taken as (top 23 bits
 * + 1/2) 2^-23, strictly inside (0, 1).  The weights are those of the
 * inverse-CDF draws: the residual max(0, p_j - q_j) (p_j where it is zero
 * everywhere), p_{L+1}, softmax(Qnew_m / T).  Both samplers draw exactly from
 * the same distributions (the Gumbel-max property), so every guarantee of
 * isd_verify_propose holds; the tokens differ because the random numbers
 * differ.  Ratios, accept lengths, alpha, greedy (T = 0) tokens and valid
 * are those of isd_verify_propose.  Arguments and workspace as
 * isd_verify_propose.
 */
ISD_API isd_status isd_verify_propose_gumbel(const void* p_logits, int64_t ld_p, const void* q_logits,
                                             int64_t ld_q, isd_dtype dtype, int vocab, const int32_t* tokens,
                                             const int32_t* seq_offsets, int num_seqs, int total_positions,
                                             const float* temperature, uint64_t seed, uint64_t offset, float tau,
                                             int32_t* accept_len, int32_t* out_tokens, float* ratio, float* alpha,
                                             const void* qnew_logits, int64_t ld_qnew, int32_t* proposals,
                                             uint8_t* valid, void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of workspace isd_propose needs for this batch shape. */
ISD_API size_t isd_propose_workspace_bytes(int num_seqs, int total_positions, int vocab, isd_dtype dtype);

/*
 * isd_propose — draw the next stride's proposals from this forward's
 * mask-position logits (§3.2: the mask positions of a forward give the next
 * proposals; §3.3: argmax proposals at T = 0).
 *
 * y_m = draw from softmax(Qnew_m / T_i) with the PROPOSE uniform of position
 * m (T = 0: argmax), for m = 1..L_i.  If accept_len_or_null is given, a
 * sequence with accept_len[i] != L_i gets no proposals (valid[i] = 0,
 * proposals -1, its rows are not read): after a rejection the next step is
 * proposal-only (§3.2), so these proposals would be discarded.
 *
 * qnew_logits [total, ld] bf16 or fp32; row seq_offsets[i] + (m-1) is Qnew_m
 * proposals   [total] int32 out
 * valid       [C] uint8 out   1 if the sequence's proposals were drawn
 */
ISD_API isd_status isd_propose(const void* qnew_logits, int64_t ld, isd_dtype dtype, int vocab,
                               const int32_t* seq_offsets, int num_seqs, int total_positions,
                               const float* temperature, uint64_t seed, uint64_t offset,
                               const int32_t* accept_len_or_null, int32_t* proposals, uint8_t* valid,
                               void* workspace, size_t workspace_bytes, void* stream);

/*
 * isd_alpha — introspective acceptance rate from per-position ratios (§2):
 * alpha_per_seq[i] = mean of ratio[seq_offsets[i] .. seq_offsets[i+1]-1]
 * (NaN for an empty sequence), *alpha_mean = mean over the C sequences.
 * ratio [total] float, alpha_per_seq [C] float out, alpha_mean [1] float out.
 * Needs no workspace.
 */
ISD_API isd_status isd_alpha(const float* ratio, const int32_t* seq_offsets, int num_seqs,
                     int total_positions, float* alpha_per_seq, float* alpha_mean, void* stream);

/*
 * isd_verify_noalloc — isd_verify for callers that cannot allocate device
 * memory.  The method has no counterpart of this call; it exists for hosts
 * that are given only the logits and output buffers and may not call
 * cudaMalloc themselves: a plug-in running inside another engine's memory
 * pool, code that runs while an allocator is locked or being resized, or a
 * caller that must not add to the device's memory use per request.
 *
 * Arguments, layout, outputs and results are those of isd_verify, without
 * the workspace.  The scratch is a fixed array of ISD_NOALLOC_SCRATCH_BYTES
 * inside the library, reserved in every CUDA context that loads the library
 * until that context is destroyed.  The call allocates nothing: every
 * argument check of isd_verify comes first (a refused call touches neither
 * the array nor the stream), then it clears the part of the array the batch
 * needs (cudaMemsetAsync on `stream`) and runs isd_verify's kernels on it.
 *
 * Limits and rules:
 *   - a batch whose isd_verify_workspace_bytes() exceeds
 *     ISD_NOALLOC_SCRATCH_BYTES returns ISD_ERR_WORKSPACE and launches
 *     nothing (isd_verify_workspace_bytes() gives any batch's need: rows of
 *     V = 151936 at C = 256, L = 16 need 2,522,368 bytes in bf16, about 30 %
 *     of the array, and 4,930,816 bytes in fp32, about 59 %);
 *   - the array's device address is looked up once per CUDA context, on the
 *     first call made in it; make that first call before any stream capture;
 *   - every call on a device shares the one array: two calls that can
 *     overlap on the GPU (different streams without an event between them)
 *     race and give wrong results.  Order them, or use isd_verify with
 *     workspaces of your own.
 */
#define ISD_NOALLOC_SCRATCH_BYTES (8u << 20)
ISD_API isd_status isd_verify_noalloc(const void* p_logits, int64_t ld_p, const void* q_logits, int64_t ld_q,
                                      isd_dtype dtype, int vocab, const int32_t* tokens,
                                      const int32_t* seq_offsets, int num_seqs, int total_positions,
                                      const float* temperature, uint64_t seed, uint64_t offset,
                                      int32_t* accept_len, int32_t* out_tokens, float* ratio,
                                      float* alpha, void* stream);

/* Static, human-readable name of a status code. */
ISD_API const char* isd_status_string(isd_status status);

#ifdef __cplusplus
}
#endif

#endif /* ISD_H_ */
