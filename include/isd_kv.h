/*
 * isd_kv.h — C ABI of libisd's KV-slot commit: the cache bookkeeping of the
 * stationary-batch loop that runs ISD ("Introspective Diffusion Language
 * Models | Summary", §3.3 I-DLM Serving Stack: KV slots are allocated with a
 * batched scatter, and the entries of rejected proposals and of mask
 * positions are trimmed; which entries stay and what the next forward
 * verifies follow §3.2 Introspective Strided Decoding).
 *
 * The conventions of include/isd.h hold: device pointers owned by the
 * caller, nothing allocated, nothing synchronised, one launch on `stream`.
 */
#ifndef ISD_KV_H_
#define ISD_KV_H_

#include "isd.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Status bits of a refused commit (written to *status). */
#define ISD_KV_ERR_STATE 1
#define ISD_KV_ERR_ACCEPT 2
#define ISD_KV_ERR_SLOT 4
#define ISD_KV_ERR_POOL 8
#define ISD_KV_ERR_CAPACITY 16

/* Largest batch one commit takes. */
#define ISD_KV_MAX_SEQS (1 << 24)

/*
 * isd_kv_commit — one commit of the stationary batch after a forward and its
 * verification; the caller enqueues it after the step's isd_verify (or
 * isd_verify_propose) on the same stream.
 *
 * Cache model.  A pool of pool_size KV slots of one token each, and per
 * sequence i a row table[i][0..ld) of slot ids by position (-1 where empty).
 * Positions 0 .. seq_len[i]-1 are committed.  The forward in flight wrote
 * alloc[i] entries at positions seq_len[i] .. seq_len[i]+alloc[i]-1, in the
 * order: x_last (the newest emitted token, not cached before), the pend[i]
 * pending proposals x_1..x_L under verification, then the M = num_masks mask
 * positions.  Free slots form a stack free_slots[0 .. *free_top), top last.
 *
 * Per sequence, a = accept_len[i] (read only when L = pend[i] > 0: the
 * sequence's isd_verify accept length, indexed by batch position):
 *   alloc[i] = 0      admitted, nothing in flight (pend[i] must be 0): keeps
 *                     nothing, and its next forward is a proposal-only step;
 *   alloc[i] = 1+L+M  keeps x_last and x_1..x_a (1 + a entries; 1 when
 *                     L = 0) and trims the rejected proposals and all M mask
 *                     entries; its next forward verifies L' = M proposals
 *                     (the masks' proposals) if L = 0 or a = L, else L' = 0
 *                     (proposal-only after a rejection, §3.2);
 *   then 1 + L' + M slots are allocated right after the kept entries, and
 *   seq_len[i] += kept, pend[i] = L', alloc[i] = 1 + L' + M.
 * Trimmed slots are pushed on the stack in (sequence, position) order and
 * their table entries set to -1; the batch then takes the top sum(1+L'+M)
 * stack entries as one block, sequence i receiving the block's entries from
 * its exclusive prefix of the counts onward, in position order (the slots
 * just trimmed are the first reused).
 *
 * Arguments: int32 device arrays table [num_seqs, ld] row-major;
 * seq_len, pend, alloc, accept_len [num_seqs]; free_slots [pool_size];
 * free_top [1]; status [1] (out).  num_masks in [0, ISD_MAX_STRIDE - 1]
 * (stride N = num_masks + 1), ld >= 1, pool_size >= 0,
 * 0 <= num_seqs <= ISD_KV_MAX_SEQS.  The per-sequence arrays of an empty
 * batch, and free_slots of an empty pool, may be NULL.
 *
 * All or nothing.  *status = 0: every array above was updated.  Otherwise
 * *status is the OR of ISD_KV_ERR_* bits and no array changed:
 *   per sequence, the first of STATE (a negative field, in-flight entries
 *   past the row, alloc neither 0 nor 1+L+M, alloc 0 with L > 0) and ACCEPT
 *   (a outside [0, L]); else SLOT (a trimmed entry outside [0, pool_size))
 *   and CAPACITY (the next allocation would run past the row);
 *   then, only if no bit is set: STATE when *free_top lies outside
 *   [0, pool_size] or the pushes would overrun the pool, else POOL when the
 *   stack cannot supply the batch.
 * Host-side checks return ISD_ERR_INVALID_ARG (a required pointer NULL, ld,
 * pool_size or num_seqs negative or zero where not allowed, num_masks out of
 * range) or ISD_ERR_UNSUPPORTED (num_seqs above ISD_KV_MAX_SEQS) and launch
 * nothing.  No workspace; the kernel never waits.
 */
ISD_API isd_status isd_kv_commit(int32_t* table, int64_t ld, int32_t* seq_len, int32_t* pend, int32_t* alloc,
                                 int32_t* free_slots, int32_t* free_top, int pool_size,
                                 const int32_t* accept_len, int num_seqs, int num_masks, int32_t* status,
                                 void* stream);

#ifdef __cplusplus
}
#endif

#endif /* ISD_KV_H_ */
