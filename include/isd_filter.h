/*
 * isd_filter.h — C ABI of libisd's filtered verify and propose: the ISD step
 * under the sampling filters of the pages' evaluation setting
 * ("Introspective Diffusion Language Models | Summary", experiments §4.1:
 * temperature 1.0, top-k 50, top-p 0.95), applied to the anchor p and the
 * proposal q alike before the ratio, the residual and every draw.
 *
 * The conventions of include/isd.h hold: device pointers owned by the
 * caller, the row layout of p, q and qnew, temperatures, Philox uniforms and
 * their counters, inverse-CDF draws in vocabulary order, the validity rules
 * and the outputs of invalid sequences.  The workspaces here need no
 * clearing: every call writes what it reads.
 *
 * The filter of one row at temperature T > 0, with p = softmax(row / T):
 *   keep the top_k ids of highest probability (lower id first among equal
 *   probabilities); of those, in the same order, keep the shortest prefix
 *   whose probability, renormalised over the top_k, adds up to at least
 *   top_p; p~ = the kept probabilities renormalised, 0 elsewhere.
 * Then ratio_k = min(1, p~_k(x_k) / q~_k(x_k)), or 1 where q~_k(x_k) = 0;
 * the correction is drawn from normalize(max(0, p~_j - q~_j)) (from p~_j if
 * that is all zero), the bonus from p~_{L+1}, proposals from q~new.
 * Temperature 0 (greedy) is unaffected by the filters: argmaxes, as in
 * isd_verify and isd_propose.
 *
 * Every call runs two kernels on `stream`: a top-k selection over each row
 * it reads (one CTA per row, the row's k best (logit, id) pairs into the
 * workspace), then one warp per sequence that applies the filter and takes
 * every decision from those lists alone.  The rows are read once.
 */
#ifndef ISD_FILTER_H_
#define ISD_FILTER_H_

#include "isd.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Largest top_k the filtered calls take (the pages' setting is 50). */
#define ISD_FILTER_MAX_TOP_K 64

/* Bytes of workspace isd_verify_filtered needs: 8 * top_k bytes for each of
 * the total + C anchor rows and total proposal rows, rounded to 256; 0 for a
 * bad shape or top_k outside [1, ISD_FILTER_MAX_TOP_K]. */
ISD_API size_t isd_verify_filtered_workspace_bytes(int num_seqs, int total_positions, int top_k);

/*
 * isd_verify_filtered — isd_verify under the top-k / top-p filters above.
 * Arguments and outputs as isd_verify, plus:
 *   top_k   in [1, ISD_FILTER_MAX_TOP_K] (values above vocab keep every id)
 *   top_p   in (0, 1] (1 keeps all top_k ids)
 * Bad top_k or top_p return ISD_ERR_INVALID_ARG.  The workspace must be at
 * least isd_verify_filtered_workspace_bytes() and 256-byte aligned; it needs
 * no clearing.  The rows of p are all read, and those of q (q is read for
 * every row, whatever the sequence's temperature).
 */
ISD_API isd_status isd_verify_filtered(const void* p_logits, int64_t ld_p, const void* q_logits, int64_t ld_q,
                                       isd_dtype dtype, int vocab, const int32_t* tokens,
                                       const int32_t* seq_offsets, int num_seqs, int total_positions,
                                       const float* temperature, uint64_t seed, uint64_t offset, int top_k,
                                       float top_p, int32_t* accept_len, int32_t* out_tokens, float* ratio,
                                       float* alpha, void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of workspace isd_propose_filtered needs: 8 * top_k bytes per qnew
 * row, rounded to 256; 0 for a bad shape or top_k. */
ISD_API size_t isd_propose_filtered_workspace_bytes(int num_seqs, int total_positions, int top_k);

/*
 * isd_propose_filtered — isd_propose with every draw from the filtered
 * q~new (argmax at T = 0).  Arguments and outputs as isd_propose, plus
 * top_k and top_p as in isd_verify_filtered.  Every qnew row is read.
 */
ISD_API isd_status isd_propose_filtered(const void* qnew_logits, int64_t ld, isd_dtype dtype, int vocab,
                                        const int32_t* seq_offsets, int num_seqs, int total_positions,
                                        const float* temperature, uint64_t seed, uint64_t offset, int top_k,
                                        float top_p, const int32_t* accept_len_or_null, int32_t* proposals,
                                        uint8_t* valid, void* workspace, size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* ISD_FILTER_H_ */
