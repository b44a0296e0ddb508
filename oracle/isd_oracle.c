/*
 * isd_oracle.c — fp64 CPU oracle for the verify-and-propose step of
 * Introspective Strided Decoding (ISD).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke entry point and
 * the benchmark's CPU-baseline leg may load this library.  The product path
 * (libisd.so) neither links nor calls it, and it shares no code with it.
 *
 * It is a plain, slow restatement of what the step computes, in double
 * precision, written from "Introspective Diffusion Language Models | Summary":
 *   - §2 Background and Motivation: the introspective acceptance rate
 *       alpha = (1/L) sum_k min(1, p_k(x_k) / q_k(x_k)),
 *     where q_k produced x_k and p_k scores x_k once it is revealed.
 *   - §3.2 Introspective Strided Decoding: each proposal is accepted with
 *     probability min(1, p_k(x_k)/q_k(x_k)); at the first rejection a token is
 *     drawn from normalize(max(0, p_k - q_k)) and the later proposals are
 *     dropped; if every proposal passes, one more token is drawn from the
 *     final causal anchor.
 *   - §3.3 I-DLM Serving Stack: argmax proposals with strict verification
 *     (the greedy, temperature-0 rule: accept while x_k is the argmax of p_k).
 *   - §3.1 Introspective-Consistency Training: logits[i] predict token[i+1]
 *     (next-token shift), which fixes which logit row scores which token.
 *   - §3.3 I-DLM Serving Stack, the fused verification kernel: Gumbel-max
 *     correction draws (oracle_gumbel_*, next to the uniforms below), an
 *     exact sampler of the same distributions as the inverse-CDF draws.
 *   - §3.3 I-DLM Serving Stack, the stationary-batch loop: KV slots are
 *     allocated with a batched scatter, and the entries of rejected
 *     proposals and of mask positions are trimmed after verification
 *     (oracle_kv_commit, at the end of this file).
 *
 * Where the pages are silent the plainest reading is taken (listed in the
 * design notes): inverse-CDF sampling in vocabulary order with counter-based
 * uniforms, temperature applied to p and q alike, argmax ties go to the lowest
 * id, alpha averages over all L positions, an all-zero residual falls back to
 * p itself.
 *
 * Uniforms come from Philox4x64-10 (Salmon, Moraes, Dror, Shaw, "Parallel
 * random numbers: as easy as 1, 2, 3", SC'11), written here from that paper's
 * definition of the round function and key schedule.
 *
 * Nothing is blocked, fused or reordered beyond the definitions: every sum
 * runs in vocabulary order in double precision.
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_API __attribute__((visibility("default")))

enum { DTYPE_BF16 = 0, DTYPE_F32 = 1 };
enum { TAG_ACCEPT = 0, TAG_CORRECT = 1, TAG_BONUS = 2, TAG_PROPOSE = 3 };
enum { MAX_STRIDE = 32 };

/* ------------------------------------------------------------------------ */
/* Philox4x64-10 (Salmon et al., SC'11, section 4, the Philox family).       */
/* ------------------------------------------------------------------------ */

static void mulhilo64(uint64_t a, uint64_t b, uint64_t* hi, uint64_t* lo) {
    unsigned __int128 prod = (unsigned __int128)a * (unsigned __int128)b;
    *hi = (uint64_t)(prod >> 64);
    *lo = (uint64_t)prod;
}

/* One call: 10 rounds of the 4x64 Philox bijection keyed by `key`. */
ORACLE_API void oracle_philox4x64_10(const uint64_t ctr[4], const uint64_t key[2], uint64_t out[4]) {
    const uint64_t M0 = 0xD2E7470EE14C6C93ULL, M1 = 0xCA5A826395121157ULL;
    const uint64_t W0 = 0x9E3779B97F4A7C15ULL, W1 = 0xBB67AE8584CAA73BULL;
    uint64_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
    uint64_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) { k0 += W0; k1 += W1; }
        uint64_t hi0, lo0, hi1, lo1;
        mulhilo64(M0, x0, &hi0, &lo0);
        mulhilo64(M1, x2, &hi1, &lo1);
        uint64_t y0 = hi1 ^ x1 ^ k0;
        uint64_t y1 = lo1;
        uint64_t y2 = hi0 ^ x3 ^ k1;
        uint64_t y3 = lo0;
        x0 = y0; x1 = y1; x2 = y2; x3 = y3;
    }
    out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

/* The uniform a decision draws: counter (offset, sequence, position, purpose),
 * key (seed, 0); the top 24 bits of output word 0 scaled by 2^-24, so u lies
 * in [0, 1) and is exact in both float and double. */
ORACLE_API double oracle_uniform(uint64_t seed, uint64_t offset, uint64_t seq, uint64_t pos, uint64_t tag) {
    uint64_t ctr[4] = {offset, seq, pos, tag};
    uint64_t key[2] = {seed, 0};
    uint64_t out[4];
    oracle_philox4x64_10(ctr, key, out);
    return (double)(out[0] >> 40) * (1.0 / 16777216.0);
}

/* ------------------------------------------------------------------------ */
/* Gumbel-max draws (the sampler of the pages' fused verification kernel,   */
/* §3.3): the id maximising log w_v + g_v, g_v = -log(-log u_v) i.i.d.      */
/* standard Gumbel noise, is distributed as w / sum(w) (the Gumbel-max      */
/* property).                                                               */
/* ------------------------------------------------------------------------ */

enum { GUMBEL_TAG_BASE = 16, GUMBEL_IDS_PER_BLOCK = 4 };

/* The uniform of vocabulary id v in one Gumbel-max draw: counter (offset,
 * sequence, position, 16 + purpose + 256 * (v / 4)), key (seed, 0), output
 * word v % 4; u = (top 23 bits + 1/2) * 2^-23, strictly inside (0, 1) and
 * exact in float and double. */
ORACLE_API double oracle_gumbel_uniform(uint64_t seed, uint64_t offset, uint64_t seq, uint64_t pos, uint64_t tag,
                                        uint64_t v) {
    uint64_t ctr[4] = {offset, seq, pos, GUMBEL_TAG_BASE + tag + 256 * (v / GUMBEL_IDS_PER_BLOCK)};
    uint64_t key[2] = {seed, 0};
    uint64_t out[4];
    oracle_philox4x64_10(ctr, key, out);
    return ((double)(out[v % GUMBEL_IDS_PER_BLOCK] >> 41) + 0.5) * (1.0 / 8388608.0);
}

/* Gumbel-max draw over weights w (w_v > 0 take part): the id of the largest
 * log w_v - log(-log u_v), the lower id on ties; -1 if no weight is
 * positive.  `margin` (optional) receives the gap between the best and the
 * second-best score (+inf with one candidate). */
ORACLE_API int oracle_gumbel_draw(const double* w, int V, uint64_t seed, uint64_t offset, uint64_t seq,
                                  uint64_t pos, uint64_t tag, double* margin) {
    int best = -1;
    double top = -INFINITY, second = -INFINITY;
    for (int v = 0; v < V; ++v) {
        if (!(w[v] > 0.0)) continue;
        double u = oracle_gumbel_uniform(seed, offset, seq, pos, tag, (uint64_t)v);
        double score = log(w[v]) - log(-log(u));
        if (score > top) {
            second = top;
            top = score;
            best = v;
        } else if (score > second) {
            second = score;
        }
    }
    if (margin) *margin = best < 0 ? 0.0 : top - second;
    return best;
}

/* ------------------------------------------------------------------------ */
/* Row-level definitions over double logits.                                */
/* ------------------------------------------------------------------------ */

/* Lowest vocabulary id holding the largest logit. */
ORACLE_API int oracle_argmax(const double* logits, int V) {
    int best = 0;
    for (int v = 1; v < V; ++v)
        if (logits[v] > logits[best]) best = v;
    return best;
}

/* softmax(logits / T), T > 0, in double. */
ORACLE_API void oracle_softmax(const double* logits, int V, double T, double* out) {
    double zmax = -INFINITY;
    for (int v = 0; v < V; ++v) {
        double z = logits[v] / T;
        if (z > zmax) zmax = z;
    }
    double total = 0.0;
    for (int v = 0; v < V; ++v) {
        out[v] = exp(logits[v] / T - zmax);
        total += out[v];
    }
    for (int v = 0; v < V; ++v) out[v] /= total;
}

/* log softmax(logits / T)[x], T > 0. */
ORACLE_API double oracle_log_softmax_at(const double* logits, int V, double T, int x) {
    double zmax = -INFINITY;
    for (int v = 0; v < V; ++v) {
        double z = logits[v] / T;
        if (z > zmax) zmax = z;
    }
    double total = 0.0;
    for (int v = 0; v < V; ++v) total += exp(logits[v] / T - zmax);
    return logits[x] / T - zmax - log(total);
}

/* The sampling filters of the pages' evaluation setting (experiments, §4.1:
 * temperature 1.0, top-k 50, top-p 0.95) on one row, T > 0: p = softmax(logits/T);
 * keep the top_k ids of highest probability (lower id first among equal
 * probabilities; top_k <= 0 keeps every id); of those, in the same order,
 * keep the shortest prefix whose probability, renormalised over the top_k,
 * adds up to at least top_p (top_p >= 1 keeps them all); out = the kept
 * probabilities renormalised, 0 elsewhere.  `cut_margin` (optional) receives
 * how far the top-p cut is from moving: the smaller of (running share at the
 * last kept id - top_p) and (top_p - running share one id earlier); +inf
 * when top_p >= 1. */
typedef struct { double p; int id; } ranked_id;

static int by_rank(const void* a, const void* b) {
    const ranked_id* x = (const ranked_id*)a;
    const ranked_id* y = (const ranked_id*)b;
    if (x->p != y->p) return x->p > y->p ? -1 : 1;
    return x->id - y->id;
}

ORACLE_API void oracle_filtered_probs(const double* logits, int V, double T, int top_k, double top_p,
                                      double* out, double* cut_margin) {
    oracle_softmax(logits, V, T, out);
    ranked_id* r = (ranked_id*)malloc(sizeof(ranked_id) * (size_t)V);
    for (int v = 0; v < V; ++v) { r[v].p = out[v]; r[v].id = v; }
    qsort(r, (size_t)V, sizeof(ranked_id), by_rank);
    int kept = (top_k > 0 && top_k < V) ? top_k : V;
    double sk = 0.0;
    for (int j = 0; j < kept; ++j) sk += r[j].p;
    int n = kept;
    double margin = INFINITY;
    if (top_p < 1.0) {
        double cum = 0.0, prev = 0.0;
        for (int j = 0; j < kept; ++j) {
            prev = cum;
            cum += r[j].p / sk;
            if (cum >= top_p) { n = j + 1; break; }
        }
        margin = cum - top_p;
        if (n > 1 && top_p - prev < margin) margin = top_p - prev;
    }
    if (cut_margin) *cut_margin = margin;
    double total = 0.0;
    for (int j = 0; j < n; ++j) total += r[j].p;
    for (int v = 0; v < V; ++v) out[v] = 0.0;
    for (int j = 0; j < n; ++j) out[r[j].id] = r[j].p / total;
    free(r);
}

/* Acceptance ratio of a proposed token x (§2 and §3.2):
 *   T > 0: min(1, p(x)/q(x)) with p = softmax(P/T), q = softmax(Q/T);
 *          q(x) = 0 (log q(x) = -inf) gives 1.
 *   T = 0: the proposal mechanism is an argmax, so the ratio is the indicator
 *          that x is the (lowest-id) argmax of P; Q is not consulted (§3.3). */
ORACLE_API double oracle_ratio(const double* P, const double* Q, int V, double T, int x) {
    if (T == 0.0) return x == oracle_argmax(P, V) ? 1.0 : 0.0;
    double lp = oracle_log_softmax_at(P, V, T, x);
    double lq = oracle_log_softmax_at(Q, V, T, x);
    if (lq == -INFINITY) return 1.0;
    double r = exp(lp - lq);
    return r < 1.0 ? r : 1.0;
}

/* The acceptance test of the relaxed-acceptance ablation (Table 4 of the
 * pages' experiments: the ratio multiplied by 1 + tau): min(1, (1+tau) p(x)/q(x)).
 * tau = 0 gives the strict ratio; at T = 0 the argmax indicator stands. */
ORACLE_API double oracle_ratio_relaxed(const double* P, const double* Q, int V, double T, int x, double tau) {
    if (T == 0.0) return x == oracle_argmax(P, V) ? 1.0 : 0.0;
    const double log_px = oracle_log_softmax_at(P, V, T, x), log_qx = oracle_log_softmax_at(Q, V, T, x);
    if (log_qx == -INFINITY) return 1.0;
    return fmin(1.0, (1.0 + tau) * exp(log_px - log_qx));
}

/* Residual weights at a rejection (§3.2): w = max(0, p - q) with p, q the
 * temperature-T softmaxes; left unnormalised (sampling normalises).  If every
 * weight is zero (possible only by rounding) the weights fall back to p. */
ORACLE_API void oracle_residual(const double* P, const double* Q, int V, double T, double* w) {
    double* pp = (double*)malloc(sizeof(double) * (size_t)V);
    double* qq = (double*)malloc(sizeof(double) * (size_t)V);
    oracle_softmax(P, V, T, pp);
    oracle_softmax(Q, V, T, qq);
    double total = 0.0;
    for (int v = 0; v < V; ++v) {
        double d = pp[v] - qq[v];
        w[v] = d > 0.0 ? d : 0.0;
        total += w[v];
    }
    if (total == 0.0)
        for (int v = 0; v < V; ++v) w[v] = pp[v];
    free(pp);
    free(qq);
}

/* Inverse-CDF draw in vocabulary order: with S = sum w and t = u*S, the
 * smallest v whose running sum C(v) exceeds t; if rounding leaves none, the
 * largest v with w[v] > 0.  `margin` (optional) receives
 * min(t - C(v-1), C(v) - t) / S, the distance of t to the chosen interval's
 * ends relative to the total. */
ORACLE_API int oracle_icdf(const double* w, int V, double u, double* margin) {
    double S = 0.0;
    for (int v = 0; v < V; ++v) S += w[v];
    double t = u * S;
    double before = 0.0, c = 0.0;
    int chosen = -1;
    for (int v = 0; v < V; ++v) {
        c = before + w[v];
        if (c > t) { chosen = v; break; }
        before = c;
    }
    if (chosen < 0) {
        for (int v = V - 1; v >= 0; --v)
            if (w[v] > 0.0) { chosen = v; break; }
        if (margin) *margin = 0.0;
        return chosen;
    }
    if (margin) {
        double lo = t - before, hi = c - t;
        *margin = (lo < hi ? lo : hi) / S;
    }
    return chosen;
}

/* ------------------------------------------------------------------------ */
/* One sequence of the verify step, uniforms given explicitly.               */
/* ------------------------------------------------------------------------ */

/* P: (L+1) rows of V anchor logits; row k-1 scores x_k (k <= L), row L is the
 *    final anchor.  Q: L rows of proposal logits, row k-1 produced x_k.
 * u_accept[k-1]: the acceptance uniform of position k.
 * u_correct[j-1]: the uniform for a correction at position j.
 * u_bonus: the uniform for the bonus token.
 * Outputs: *accept_len = a; out_tokens[0..a-1] = x_1..x_a, out_tokens[a] =
 * the correction or bonus token, out_tokens[a+1..L] = -1; ratio[k-1];
 * *alpha; accept_margin[k-1] = |u_k - ratio_k| (T > 0; +inf when T = 0, the
 * greedy decisions compare exact logits); *token_margin = the draw's ICDF
 * margin (+inf for an argmax). */
ORACLE_API void oracle_verify_one(const double* P, const double* Q, int V, int L, double T,
                                  const int32_t* x, const double* u_accept, const double* u_correct,
                                  double u_bonus, int32_t* accept_len, int32_t* out_tokens,
                                  double* ratio, double* alpha, double* accept_margin,
                                  double* token_margin, double tau) {
    /* §2: ratios of every position, and their mean. */
    double sum = 0.0;
    for (int k = 1; k <= L; ++k) {
        ratio[k - 1] = oracle_ratio(P + (size_t)(k - 1) * V, Q + (size_t)(k - 1) * V, V, T, x[k - 1]);
        sum += ratio[k - 1];
    }
    *alpha = sum / L;

    /* §3.2: strict acceptance, the accepted prefix ends at the first rejection.
     * With tau > 0 the test uses the relaxed ratio instead; the reported
     * ratios and alpha stay the strict ones (§2). */
    int a = 0;
    for (int k = 1; k <= L; ++k) {
        int accepted;
        double racc = ratio[k - 1];
        if (tau != 0.0)
            racc = oracle_ratio_relaxed(P + (size_t)(k - 1) * V, Q + (size_t)(k - 1) * V, V, T, x[k - 1], tau);
        if (T == 0.0) {
            accepted = ratio[k - 1] == 1.0;
            accept_margin[k - 1] = INFINITY;
        } else {
            accepted = u_accept[k - 1] < racc;
            accept_margin[k - 1] = fabs(u_accept[k - 1] - racc);
        }
        if (!accepted) break;
        a = k;
    }
    /* Margins of decisions after the first rejection were never taken. */
    for (int k = a + 2; k <= L; ++k) accept_margin[k - 1] = INFINITY;

    int token;
    if (a < L) {
        /* Correction at j = a + 1 from normalize(max(0, p_j - q_j)). */
        int j = a + 1;
        const double* Pj = P + (size_t)(j - 1) * V;
        const double* Qj = Q + (size_t)(j - 1) * V;
        if (T == 0.0) {
            token = oracle_argmax(Pj, V);
            *token_margin = INFINITY;
        } else {
            double* w = (double*)malloc(sizeof(double) * (size_t)V);
            oracle_residual(Pj, Qj, V, T, w);
            token = oracle_icdf(w, V, u_correct[j - 1], token_margin);
            free(w);
        }
    } else {
        /* Bonus token from the final causal anchor p_{L+1}. */
        const double* Pb = P + (size_t)L * V;
        if (T == 0.0) {
            token = oracle_argmax(Pb, V);
            *token_margin = INFINITY;
        } else {
            double* w = (double*)malloc(sizeof(double) * (size_t)V);
            oracle_softmax(Pb, V, T, w);
            token = oracle_icdf(w, V, u_bonus, token_margin);
            free(w);
        }
    }
    *accept_len = a;
    for (int m = 0; m < a; ++m) out_tokens[m] = x[m];
    out_tokens[a] = token;
    for (int m = a + 1; m <= L; ++m) out_tokens[m] = -1;
}

/* ------------------------------------------------------------------------ */
/* Batched entry points with the library's argument meaning (host memory).   */
/* ------------------------------------------------------------------------ */

static double logit_value(const void* base, int dtype, int64_t ld, int64_t row, int64_t v) {
    if (dtype == DTYPE_F32) return (double)((const float*)base)[row * ld + v];
    /* bfloat16: the upper 16 bits of an IEEE binary32. */
    uint16_t h = ((const uint16_t*)base)[row * ld + v];
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

static void load_rows(const void* base, int dtype, int64_t ld, int64_t first_row, int nrows, int V,
                      double* out) {
    for (int r = 0; r < nrows; ++r)
        for (int v = 0; v < V; ++v)
            out[(size_t)r * V + v] = logit_value(base, dtype, ld, first_row + r, v);
}

/* T = 0 (greedy) or a finite normal positive float; subnormal temperatures
 * are rejected (log2(e)/T would overflow a float scale). */
static int temperature_ok(float T) { return isfinite(T) && (T == 0.0f || T >= FLT_MIN); }

static void set_threads(int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

/* Threads the parallel loops will use. */
ORACLE_API int oracle_max_threads(int nthreads) {
#ifdef _OPENMP
    return nthreads > 0 ? nthreads : omp_get_max_threads();
#else
    (void)nthreads;
    return 1;
#endif
}

/* Row layout (§3.1 next-token shift, one more anchor row than proposals):
 *   sequence i has L_i = seq_offsets[i+1] - seq_offsets[i] proposals;
 *   p row of position k (1..L_i+1) is seq_offsets[i] + i + k - 1;
 *   q row and token of position k (1..L_i) are seq_offsets[i] + k - 1.
 * A sequence with L_i outside [1, 32], a temperature that is negative,
 * subnormal or not finite, or a token outside [0, V) is invalid: accept_len = -1, its output
 * slots -1, its ratios and alpha NaN.
 * `seqs` (optional, n_sel entries) restricts the work to those sequences;
 * the other sequences' outputs are left untouched. */
ORACLE_API void oracle_verify(const void* p_logits, int64_t ld_p, const void* q_logits, int64_t ld_q,
                              int dtype, int V, const int32_t* tokens, const int32_t* seq_offsets,
                              int num_seqs, const float* temperature, uint64_t seed, uint64_t offset,
                              int32_t* accept_len, int32_t* out_tokens, double* ratio, double* alpha,
                              double* accept_margin, double* token_margin, const int32_t* seqs,
                              int n_sel, int nthreads, double tau) {
    set_threads(nthreads);
    int count = seqs ? n_sel : num_seqs;
#pragma omp parallel for schedule(dynamic, 1)
    for (int s = 0; s < count; ++s) {
        int i = seqs ? seqs[s] : s;
        int start = seq_offsets[i];
        int L = seq_offsets[i + 1] - start;
        float T = temperature[i];
        int valid = L >= 1 && L <= MAX_STRIDE && temperature_ok(T);
        for (int k = 0; valid && k < L; ++k)
            if (tokens[start + k] < 0 || tokens[start + k] >= V) valid = 0;
        if (!valid) {
            accept_len[i] = -1;
            alpha[i] = NAN;
            token_margin[i] = INFINITY;
            if (L >= 0) {
                for (int m = 0; m <= L; ++m) out_tokens[start + i + m] = -1;
                for (int k = 0; k < L; ++k) {
                    ratio[start + k] = NAN;
                    accept_margin[start + k] = INFINITY;
                }
            }
            continue;
        }
        double* P = (double*)malloc(sizeof(double) * (size_t)(L + 1) * V);
        double* Q = (double*)malloc(sizeof(double) * (size_t)L * V);
        load_rows(p_logits, dtype, ld_p, (int64_t)start + i, L + 1, V, P);
        load_rows(q_logits, dtype, ld_q, (int64_t)start, L, V, Q);
        double u_acc[MAX_STRIDE], u_cor[MAX_STRIDE];
        for (int k = 1; k <= L; ++k) {
            u_acc[k - 1] = oracle_uniform(seed, offset, (uint64_t)i, (uint64_t)k, TAG_ACCEPT);
            u_cor[k - 1] = oracle_uniform(seed, offset, (uint64_t)i, (uint64_t)k, TAG_CORRECT);
        }
        double u_bonus = oracle_uniform(seed, offset, (uint64_t)i, (uint64_t)(L + 1), TAG_BONUS);
        oracle_verify_one(P, Q, V, L, (double)T, tokens + start, u_acc, u_cor, u_bonus,
                          &accept_len[i], out_tokens + start + i, ratio + start, &alpha[i],
                          accept_margin + start, &token_margin[i], tau);
        free(P);
        free(Q);
    }
}

/* Proposals for the next stride (§3.2, §3.3): y_m drawn from softmax(qnew_m/T)
 * by inverse CDF with the PROPOSE uniform of position m, argmax at T = 0.
 * With accept_len given, a sequence whose proposals were not all accepted
 * (a_i != L_i) gets no proposals: after a rejection the next step is
 * proposal-only, so these would be discarded (valid = 0, proposals -1).
 * margin[row] receives the draw's ICDF margin (+inf for argmax or skipped). */
ORACLE_API void oracle_propose(const void* qnew_logits, int64_t ld, int dtype, int V,
                               const int32_t* seq_offsets, int num_seqs, const float* temperature,
                               uint64_t seed, uint64_t offset, const int32_t* accept_len_or_null,
                               int32_t* proposals, uint8_t* valid, double* margin,
                               const int32_t* seqs, int n_sel, int nthreads) {
    set_threads(nthreads);
    int count = seqs ? n_sel : num_seqs;
#pragma omp parallel for schedule(dynamic, 1)
    for (int s = 0; s < count; ++s) {
        int i = seqs ? seqs[s] : s;
        int start = seq_offsets[i];
        int L = seq_offsets[i + 1] - start;
        float T = temperature[i];
        int ok = L >= 1 && L <= MAX_STRIDE && temperature_ok(T);
        if (ok && accept_len_or_null) ok = accept_len_or_null[i] == L;
        valid[i] = (uint8_t)ok;
        if (!ok) {
            if (L >= 0)
                for (int m = 0; m < L; ++m) {
                    proposals[start + m] = -1;
                    margin[start + m] = INFINITY;
                }
            continue;
        }
        double* row = (double*)malloc(sizeof(double) * (size_t)V);
        double* w = (double*)malloc(sizeof(double) * (size_t)V);
        for (int m = 1; m <= L; ++m) {
            load_rows(qnew_logits, dtype, ld, (int64_t)start + m - 1, 1, V, row);
            if (T == 0.0f) {
                proposals[start + m - 1] = oracle_argmax(row, V);
                margin[start + m - 1] = INFINITY;
            } else {
                oracle_softmax(row, V, (double)T, w);
                double u = oracle_uniform(seed, offset, (uint64_t)i, (uint64_t)m, TAG_PROPOSE);
                proposals[start + m - 1] = oracle_icdf(w, V, u, &margin[start + m - 1]);
            }
        }
        free(row);
        free(w);
    }
}

/* alpha per sequence as the mean of its L_i ratios (§2), and the batch mean
 * of the per-sequence values. */
ORACLE_API void oracle_alpha(const float* ratio, const int32_t* seq_offsets, int num_seqs,
                             double* alpha_per_seq, double* alpha_mean) {
    double total = 0.0;
    for (int i = 0; i < num_seqs; ++i) {
        int start = seq_offsets[i];
        int L = seq_offsets[i + 1] - start;
        double s = 0.0;
        for (int k = 0; k < L; ++k) s += (double)ratio[start + k];
        alpha_per_seq[i] = L > 0 ? s / L : NAN;
        total += alpha_per_seq[i];
    }
    *alpha_mean = num_seqs > 0 ? total / num_seqs : NAN;
}

/* ------------------------------------------------------------------------ */
/* KV-slot bookkeeping of the stationary-batch loop (§3.3: slots allocated   */
/* with a batched scatter; rejected and masked entries trimmed).             */
/* ------------------------------------------------------------------------ */

enum { KV_ERR_STATE = 1, KV_ERR_ACCEPT = 2, KV_ERR_SLOT = 4, KV_ERR_POOL = 8, KV_ERR_CAPACITY = 16 };

/* Per-sequence outcome of one commit; 0 or one KV_ERR_* bit set. */
static int kv_plan(const int32_t* table_row, int64_t ld, int len, int L, int w, int a_in, int M,
                   int pool_size, int* kept, int* next_pend, int* status) {
    *status = 0;
    if (len < 0 || L < 0 || w < 0 || (int64_t)len + w > ld || (w == 0 && L != 0) ||
        (w > 0 && (int64_t)w != 1 + (int64_t)L + M)) {
        *status = KV_ERR_STATE;
        return 0;
    }
    if (w == 0) {               /* admitted, no forward in flight yet */
        *kept = 0;
        *next_pend = 0;
    } else {
        int a = L > 0 ? a_in : 0;   /* a proposal-only step verified nothing */
        if (a < 0 || a > L) {
            *status = KV_ERR_ACCEPT;
            return 0;
        }
        *kept = 1 + a;                               /* x_last, then x_1..x_a */
        *next_pend = (L == 0 || a == L) ? M : 0;     /* the masks' proposals stand */
    }
    for (int j = *kept; j < w; ++j) {
        int32_t slot = table_row[len + j];
        if (slot < 0 || slot >= pool_size) *status |= KV_ERR_SLOT;
    }
    if ((int64_t)len + *kept + 1 + *next_pend + M > ld) *status |= KV_ERR_CAPACITY;
    return 1;
}

/*
 * One commit of the stationary batch after a forward and its verification.
 *
 * Cache model: a pool of pool_size KV slots (one token each) and, per
 * sequence i, a row table[i][0..ld) of slot ids by position.  Positions
 * 0..seq_len[i]-1 are committed; the forward in flight wrote alloc[i]
 * entries at positions seq_len[i] .. seq_len[i]+alloc[i]-1, in the order
 *     x_last, the pend[i] pending proposals x_1..x_L, the M mask positions,
 * where x_last is the newest emitted token (§3.2: one anchor token, the
 * proposals under verification, then the mask positions that propose).
 * The free slots are a stack free_slots[0..*free_top), top last.
 *
 * Per sequence, with a = accept_len[i] (read only when L = pend[i] > 0):
 *   alloc = 0 (just admitted; pend must be 0): keeps nothing, and its next
 *       forward is a proposal-only step;
 *   alloc = 1 + L + M: keeps x_last and the accepted x_1..x_a (1 + a
 *       entries; 1 when L = 0), trims the rejected proposals and every mask
 *       entry (§3.3), and its next forward verifies the masks' M proposals
 *       when every proposal passed or none were pending (L' = M), else is
 *       proposal-only (L' = 0, §3.2);
 *   the next forward's 1 + L' + M entries are allocated right after the
 *       kept ones.
 * Trimmed slots are pushed on the stack in (sequence, position) order and
 * their table entries set to -1; then the batch takes the top sum(1+L'+M)
 * entries of the stack as one block, sequence i receiving the block's
 * entries from its exclusive prefix of the counts onward, in position
 * order (so the slots just trimmed are the first reused).
 *
 * Returns 0 after updating table, seq_len, pend, alloc, free_slots and
 * free_top.  Otherwise returns the OR of KV_ERR_* bits and changes nothing:
 *   per sequence, the first of STATE (negative fields, alloc past the row,
 *   alloc not 0 or 1+L+M, alloc 0 with L > 0) and ACCEPT (a outside [0, L]),
 *   else SLOT (a trimmed entry outside [0, pool_size)) and CAPACITY (the
 *   next allocation runs past the row);
 *   then, only when no bit is set: STATE if *free_top lies outside
 *   [0, pool_size] or the pushes would overrun the pool, else POOL if the
 *   stack cannot supply the batch.
 */
ORACLE_API int oracle_kv_commit(int32_t* table, int64_t ld, int32_t* seq_len, int32_t* pend, int32_t* alloc,
                                int32_t* free_slots, int32_t* free_top, int pool_size,
                                const int32_t* accept_len, int num_seqs, int num_masks) {
    int M = num_masks;
    int status = 0;
    int64_t pushed = 0, wanted = 0;
    for (int i = 0; i < num_seqs; ++i) {
        int kept, next_pend, st;
        if (kv_plan(table + (int64_t)i * ld, ld, seq_len[i], pend[i], alloc[i], accept_len[i], M, pool_size,
                    &kept, &next_pend, &st)) {
            pushed += alloc[i] - kept;
            wanted += 1 + next_pend + M;
        }
        status |= st;
    }
    if (status) return status;
    int64_t top = *free_top;
    if (top < 0 || top > pool_size || top + pushed > pool_size) return KV_ERR_STATE;
    if (top + pushed < wanted) return KV_ERR_POOL;

    /* trim: push the trimmed slots, clear their table entries */
    for (int i = 0; i < num_seqs; ++i) {
        int kept, next_pend, st;
        kv_plan(table + (int64_t)i * ld, ld, seq_len[i], pend[i], alloc[i], accept_len[i], M, pool_size,
                &kept, &next_pend, &st);
        for (int j = kept; j < alloc[i]; ++j) {
            int32_t* e = &table[(int64_t)i * ld + seq_len[i] + j];
            free_slots[top++] = *e;
            *e = -1;
        }
    }
    /* batched scatter: the top `wanted` stack entries, in sequence order */
    int64_t next = top - wanted;
    *free_top = (int32_t)next;
    for (int i = 0; i < num_seqs; ++i) {
        int kept, next_pend, st;
        kv_plan(table + (int64_t)i * ld, ld, seq_len[i], pend[i], alloc[i], accept_len[i], M, pool_size,
                &kept, &next_pend, &st);
        int n = 1 + next_pend + M;
        int len = seq_len[i] + kept;
        for (int j = 0; j < n; ++j) table[(int64_t)i * ld + len + j] = free_slots[next++];
        seq_len[i] = len;
        pend[i] = next_pend;
        alloc[i] = n;
    }
    return 0;
}
