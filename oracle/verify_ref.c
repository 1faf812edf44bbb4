/*
 * Plain fp64 CPU oracle of the speculative-sampling verify step.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or call this file:
 * only tests/, the smoke check in __graft_entry__.py and the CPU-baseline leg of bench.py use it.
 * It shares no code, header, table or constant with the CUDA library; the two agree only
 * through the published definitions they both follow.
 *
 * Sources (page titles; sections as printed on the pages):
 *   [velog]   "6-1편. Speculative Decoding" (velog article walking through Leviathan et al.)
 *             §1-2 (p and q are next-token distributions), §2 "4-step algorithm",
 *             §2-1 (accept/reject rule min(1, p/q)), §2-2 (corrected distribution
 *             p' = norm(max(0, p - q)) and "sampling" in proportion to probability),
 *             §2-3 (beta, p' = (p - min(p,q))/(1 - beta), losslessness).
 *   [scaling] "All About Transformer Inference", Appendix D "Speculative Sampling"
 *             (greedy variant, steps 1-3: accept while the draft equals the target's
 *             highest-probability token; replace the first wrong one; one extra token
 *             from the last logits when all match).
 *   [sonar]   "Accelerating Sonar through speculation", §"Speculative decoding"
 *             (n drafted tokens yield up to n + 1 emitted tokens).
 *   Philox4x32-10: Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3",
 *             SC'11 (the counter-based generator the verify step draws its uniforms from).
 *
 * Readings of points the pages leave open (each one is listed in the design notes):
 *   - p = softmax(l / T) and q = softmax(l_draft / T) with the same temperature T.
 *   - accept draft x iff u * q(x) < p(x), u uniform on [0, 1): this is "accept with probability
 *     min(1, p/q)" with q <= p always accepted; p = q = 0 rejects.
 *   - sampling "in proportion to probability" is an inverse CDF in vocabulary index order:
 *     the token is the smallest k with C_k > u * S, C_k the running sum of the weights in
 *     index order and S the total; if rounding leaves no such k, the last k with weight > 0.
 *   - the residual normaliser S is the direct sum of max(0, p - q) (equal to 1 - beta in exact
 *     arithmetic); if it is exactly 0 the draw falls back to p.
 *   - greedy (T == 0): argmax of the raw target logits, lowest index on ties.
 *   - drafts without a draft distribution (an n-gram drafter, [velog] §"drafter types": the tokens
 *     that followed an earlier occurrence of the last n tokens): no draft rows are given (draft NULL
 *     with T > 0), and q_i is the point mass at x_i. The rule above is applied unchanged: accept iff
 *     u < p(x), residual p with x removed.
 *   - uniform u = (Philox4x32-10(ctr, key).x0 >> 8) * 2^-24 with key = (lo32 seed, hi32 seed),
 *     ctr = (lo32 step, hi32 step, seq, (slot << 8) | purpose); purpose 0 = accept test of
 *     slot i, purpose 1 = residual/bonus draw at the emitting slot.
 *
 * Parity pins (tests, CPU): Philox against curand's host Philox4x32-10 generator; softmax
 * normaliser against torch.log_softmax in float64; greedy against torch.argmax; accept rule,
 * p' and beta against hand-worked cases; joint output law against exact rational enumeration;
 * beta, losslessness and E[N] statistically. The inverse-CDF tail rule, the S == 0 fallback and
 * the handling of -inf weights are conventions the pages do not fix: parity unpinned there
 * beyond unit cases.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* error codes, numbered like the library's status codes (kept separate on purpose) */
enum {
    OR_OK = 0,
    OR_ERR_INVALID_ARG = 1,
    OR_ERR_BAD_TOKEN = 3,
    OR_ERR_BAD_OFFSETS = 4,
    OR_ERR_NONFINITE = 5,
    OR_ERR_EMPTY_ROW = 6,
};
enum { OR_F32 = 0, OR_BF16 = 1 };

/* ------------------------------------------------------------------------------------------ */
/* Philox4x32-10 (Salmon et al., SC'11): 10 rounds of the 4x32 S-box with key schedule.       */
/* ------------------------------------------------------------------------------------------ */
static void philox_round(uint32_t c[4], const uint32_t k[2]) {
    const uint64_t p0 = (uint64_t)0xD2511F53u * (uint64_t)c[0];
    const uint64_t p1 = (uint64_t)0xCD9E8D57u * (uint64_t)c[2];
    const uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    const uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    uint32_t n[4];
    n[0] = hi1 ^ c[1] ^ k[0];
    n[1] = lo1;
    n[2] = hi0 ^ c[3] ^ k[1];
    n[3] = lo0;
    memcpy(c, n, sizeof n);
}

void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
    uint32_t c[4] = {ctr[0], ctr[1], ctr[2], ctr[3]};
    uint32_t k[2] = {key[0], key[1]};
    for (int r = 0; r < 10; ++r) {
        if (r > 0) { /* key bump by the Weyl constants between rounds */
            k[0] += 0x9E3779B9u;
            k[1] += 0xBB67AE85u;
        }
        philox_round(c, k);
    }
    memcpy(out, c, sizeof c);
}

double oracle_uniform(uint64_t seed, uint64_t step, uint32_t seq, uint32_t slot, uint32_t purpose) {
    const uint32_t ctr[4] = {(uint32_t)step, (uint32_t)(step >> 32), seq, (slot << 8) | (purpose & 0xFFu)};
    const uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t out[4];
    oracle_philox4x32_10(ctr, key, out);
    return (double)(out[0] >> 8) * (1.0 / 16777216.0);
}

/* ------------------------------------------------------------------------------------------ */
/* Inverse-CDF draw in vocabulary index order ([velog] §2-2 "sampling").                      */
/* ------------------------------------------------------------------------------------------ */
static int32_t invcdf(const double* w, int32_t V, double S, double u) {
    const double target = u * S;
    double c = 0.0;
    for (int32_t k = 0; k < V; ++k) {
        c += w[k];
        if (c > target) return k;
    }
    for (int32_t k = V - 1; k >= 0; --k) /* rounding left no crossing: last positive weight */
        if (w[k] > 0.0) return k;
    return -1;
}

/*
 * Core verify step on fp64 probabilities, one sequence ([velog] §2 steps 3-4, §2-1, §2-2).
 *   p: (gamma + 1) rows of V target probabilities; q: gamma rows of V draft probabilities;
 *   x: gamma draft tokens; u_acc[i]: uniform for the accept test of slot i; u_smp[i]: uniform
 *   for a draw at slot i (residual at a rejected slot, bonus at slot gamma).
 *   Writes gamma + 1 tokens (-1 after the emitting slot) and returns n, the number of accepted
 *   drafts. *mass (nullable) receives the draw's normaliser S; *fallback (nullable) is set when a
 *   rejected slot's residual mass was exactly 0 and the draw used p instead.
 */
int32_t oracle_verify_probs(const double* p, const double* q, const int32_t* x, int32_t gamma,
                            int32_t V, const double* u_acc, const double* u_smp, int32_t* out,
                            double* mass, int32_t* fallback) {
    double* w = (double*)malloc(sizeof(double) * (size_t)(V > 0 ? V : 1));
    int32_t n = gamma;
    if (fallback) *fallback = 0;
    for (int32_t i = 0; i < gamma; ++i) {
        const double* pi = p + (size_t)i * V;
        const double* qi = q + (size_t)i * V;
        const int32_t xi = x[i];
        if (u_acc[i] * qi[xi] < pi[xi]) { /* accepted with probability min(1, p/q) */
            out[i] = xi;
            continue;
        }
        /* first rejection: residual p' = norm(max(0, p - q)) */
        double S = 0.0;
        for (int32_t k = 0; k < V; ++k) {
            w[k] = pi[k] > qi[k] ? pi[k] - qi[k] : 0.0;
            S += w[k];
        }
        if (S == 0.0) { /* p' undefined (1 - beta == 0 only through rounding): draw from p */
            for (int32_t k = 0; k < V; ++k) { w[k] = pi[k]; S += w[k]; }
            if (fallback) *fallback = 1;
        }
        out[i] = invcdf(w, V, S, u_smp[i]);
        if (mass) *mass = S;
        n = i;
        break;
    }
    if (n == gamma) { /* every draft accepted: bonus token from p at slot gamma */
        const double* pg = p + (size_t)gamma * V;
        double S = 0.0;
        for (int32_t k = 0; k < V; ++k) S += pg[k];
        out[gamma] = invcdf(pg, V, S, u_smp[gamma]);
        if (mass) *mass = S;
    }
    for (int32_t j = n + 1; j <= gamma; ++j) out[j] = -1;
    free(w);
    return n;
}

/* ------------------------------------------------------------------------------------------ */
/* Logit rows -> probabilities                                                                */
/* ------------------------------------------------------------------------------------------ */
static double logit_at(const void* base, int dtype, size_t idx) {
    if (dtype == OR_BF16) {
        const uint16_t h = ((const uint16_t*)base)[idx];
        const uint32_t bits = (uint32_t)h << 16; /* bf16 -> fp32 is exact */
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f;
    }
    return (double)((const float*)base)[idx];
}

/* p = softmax(l / T) in fp64 ([velog] §1-2; temperature per the reading above). Returns an error
 * code; *lse receives log sum exp(l / T). */
static int row_softmax(const void* base, int dtype, size_t row, int32_t V, double T, double* prob,
                       double* lse) {
    double m = -INFINITY;
    for (int32_t k = 0; k < V; ++k) {
        const double l = logit_at(base, dtype, row * (size_t)V + (size_t)k);
        if (isnan(l) || l == INFINITY) return OR_ERR_NONFINITE;
        const double z = l / T;
        prob[k] = z;
        if (z > m) m = z;
    }
    if (m == -INFINITY) return OR_ERR_EMPTY_ROW;
    double s = 0.0;
    for (int32_t k = 0; k < V; ++k) {
        prob[k] = exp(prob[k] - m);
        s += prob[k];
    }
    for (int32_t k = 0; k < V; ++k) prob[k] /= s;
    if (lse) *lse = m + log(s);
    return OR_OK;
}

/* greedy argmax of raw logits, lowest index on ties ([scaling] App. D step 3) */
static int row_argmax(const void* base, int dtype, size_t row, int32_t V, int32_t* arg) {
    double m = -INFINITY;
    int32_t a = -1;
    for (int32_t k = 0; k < V; ++k) {
        const double l = logit_at(base, dtype, row * (size_t)V + (size_t)k);
        if (isnan(l) || l == INFINITY) return OR_ERR_NONFINITE;
        if (a < 0 || l > m) { m = l; a = k; }
    }
    if (m == -INFINITY) return OR_ERR_EMPTY_ROW;
    *arg = a;
    return OR_OK;
}

typedef struct {
    double* row_lse;      /* [R_t + R_d] log sum exp(l / T): target rows first, then draft rows */
    int32_t* row_argmax;  /* [R_t] greedy argmax of each target row (greedy mode only) */
    double* p_x;          /* [R_d] p_i(x_i) of every draft slot */
    double* q_x;          /* [R_d] q_i(x_i) of every draft slot */
    double* seq_mass;     /* [B] normaliser S of the sequence's draw */
    int32_t* seq_fallback;/* [B] 1 where the S == 0 fallback was taken */
    double* beta;         /* [R_d] beta_i = sum_x min(p_i(x), q_i(x)) of every draft slot ([velog] §2-3) */
} oracle_debug;

typedef struct {
    const void* target;
    const void* draft;
    int dtype;
    const int32_t* tok;
    const int32_t* off;
    const int32_t* gam;
    int32_t B, V;
    double T;
    uint64_t seed, step;
    int32_t* out_tok;
    int32_t* out_n;
    oracle_debug* dbg;
    int32_t b0, b1;
    int32_t nsteps;   /* sampling mode: draws for steps step .. step + nsteps - 1 (outputs step-major) */
    uint32_t seq_base;/* global index of sequence 0: sequence b's uniforms are keyed by seq_base + b */
    uint32_t status;
} job_t;

static void fail_seq(job_t* J, int32_t b, int code) {
    const int32_t d0 = J->off[b], g = J->gam[b];
    const size_t R_t = (size_t)J->off[J->B] + (size_t)J->B;
    const int32_t ns = J->T == 0.0 ? 1 : J->nsteps;
    for (int32_t s = 0; s < ns; ++s) {
        for (int32_t j = 0; j <= g; ++j) J->out_tok[(size_t)s * R_t + (size_t)(d0 + b + j)] = -1;
        J->out_n[(size_t)s * (size_t)J->B + b] = -1;
    }
    J->status |= 1u << code;
}

static void verify_one(job_t* J, int32_t b, double* prow, double* qrow, double* u_acc,
                       double* u_smp) {
    const int32_t V = J->V;
    const int32_t g = J->gam[b];
    const int32_t d0 = J->off[b];
    const int32_t t0 = d0 + b;
    const int32_t R_t = J->off[J->B] + J->B;
    const int32_t* x = J->tok + d0;
    for (int32_t i = 0; i < g; ++i)
        if (x[i] < 0 || x[i] >= V) { fail_seq(J, b, OR_ERR_BAD_TOKEN); return; }

    if (J->T == 0.0) { /* greedy ([scaling] App. D steps 1-3) */
        int32_t n = g;
        for (int32_t i = 0; i <= g; ++i) {
            int32_t a;
            const int e = row_argmax(J->target, J->dtype, (size_t)(t0 + i), V, &a);
            if (e) { fail_seq(J, b, e); return; }
            if (J->dbg && J->dbg->row_argmax) J->dbg->row_argmax[t0 + i] = a;
            if (i < n) {
                J->out_tok[t0 + i] = a;
                if (i < g && x[i] != a) n = i; /* first wrong draft replaced by the argmax */
            } else if (i == n) {
                J->out_tok[t0 + i] = a;
            }
        }
        for (int32_t j = n + 1; j <= g; ++j) J->out_tok[t0 + j] = -1;
        J->out_n[b] = n;
        return;
    }

    for (int32_t i = 0; i <= g; ++i) {
        double lse;
        int e = row_softmax(J->target, J->dtype, (size_t)(t0 + i), V, J->T, prow + (size_t)i * V, &lse);
        if (e) { fail_seq(J, b, e); return; }
        if (J->dbg && J->dbg->row_lse) J->dbg->row_lse[t0 + i] = lse;
        if (i < g && !J->draft) { /* point-mass draft: q_i = 1 at x_i, 0 elsewhere */
            double* qi = qrow + (size_t)i * V;
            for (int32_t k = 0; k < V; ++k) qi[k] = 0.0;
            qi[x[i]] = 1.0;
            if (J->dbg && J->dbg->p_x) J->dbg->p_x[d0 + i] = prow[(size_t)i * V + x[i]];
            if (J->dbg && J->dbg->q_x) J->dbg->q_x[d0 + i] = 1.0;
            if (J->dbg && J->dbg->beta) J->dbg->beta[d0 + i] = prow[(size_t)i * V + x[i]]; /* min(p, 1{x}) */
        } else if (i < g) {
            e = row_softmax(J->draft, J->dtype, (size_t)(d0 + i), V, J->T, qrow + (size_t)i * V, &lse);
            if (e) { fail_seq(J, b, e); return; }
            if (J->dbg && J->dbg->row_lse) J->dbg->row_lse[R_t + d0 + i] = lse;
            if (J->dbg && J->dbg->p_x) J->dbg->p_x[d0 + i] = prow[(size_t)i * V + x[i]];
            if (J->dbg && J->dbg->q_x) J->dbg->q_x[d0 + i] = qrow[(size_t)i * V + x[i]];
            if (J->dbg && J->dbg->beta) { /* [velog] §2-3: beta = sum_x min(p(x), q(x)) */
                const double* pi = prow + (size_t)i * V;
                const double* qi = qrow + (size_t)i * V;
                double bsum = 0.0;
                for (int32_t k = 0; k < V; ++k) bsum += pi[k] < qi[k] ? pi[k] : qi[k];
                J->dbg->beta[d0 + i] = bsum;
            }
        }
    }
    /* the draws of this step and of every further step the job asks for: the same rule on the same
       probabilities, with the uniforms of step + s (multi-step verification of one batch) */
    for (int32_t s = 0; s < J->nsteps; ++s) {
        const uint64_t step = J->step + (uint64_t)s;
        for (int32_t i = 0; i <= g; ++i) {
            u_acc[i] = oracle_uniform(J->seed, step, J->seq_base + (uint32_t)b, (uint32_t)i, 0);
            u_smp[i] = oracle_uniform(J->seed, step, J->seq_base + (uint32_t)b, (uint32_t)i, 1);
        }
        double S = 0.0;
        int32_t fb = 0;
        int32_t* out_tok = J->out_tok + (size_t)s * (size_t)R_t;
        const int32_t n = oracle_verify_probs(prow, qrow, x, g, V, u_acc, u_smp, out_tok + t0, &S, &fb);
        J->out_n[(size_t)s * (size_t)J->B + b] = n;
        if (s == 0 && J->dbg && J->dbg->seq_mass) J->dbg->seq_mass[b] = S;
        if (s == 0 && J->dbg && J->dbg->seq_fallback) J->dbg->seq_fallback[b] = fb;
    }
}

static void* run_job(void* arg) {
    job_t* J = (job_t*)arg;
    int32_t gmax = 0;
    for (int32_t b = J->b0; b < J->b1; ++b) gmax = J->gam[b] > gmax ? J->gam[b] : gmax;
    const size_t V = (size_t)J->V;
    double* prow = (double*)malloc(sizeof(double) * V * (size_t)(gmax + 1));
    double* qrow = (double*)malloc(sizeof(double) * V * (size_t)(gmax > 0 ? gmax : 1));
    double* u_acc = (double*)malloc(sizeof(double) * (size_t)(gmax + 1));
    double* u_smp = (double*)malloc(sizeof(double) * (size_t)(gmax + 1));
    for (int32_t b = J->b0; b < J->b1; ++b) verify_one(J, b, prow, qrow, u_acc, u_smp);
    free(prow); free(qrow); free(u_acc); free(u_smp);
    return NULL;
}

/*
 * Verify a CSR-packed batch: sequence b has gammas[b] draft rows seq_offsets[b] ..
 * seq_offsets[b+1]-1 and gammas[b] + 1 target rows seq_offsets[b] + b .. seq_offsets[b+1] + b.
 * All arrays are host arrays. Returns the OR of (1 << error code) over all sequences (0 = OK);
 * a failed sequence gets n = -1 and tokens -1. Batch-level argument errors return
 * 1 << OR_ERR_INVALID_ARG or 1 << OR_ERR_BAD_OFFSETS without touching the outputs.
 */
static uint32_t verify_batch(const void* target, const void* draft, int dtype, const int32_t* draft_tokens,
                             const int32_t* seq_offsets, const int32_t* gammas, int32_t B, int32_t V,
                             double temperature, uint64_t seed, uint64_t step, uint32_t seq_base, int32_t nsteps,
                             int32_t* out_tokens, int32_t* out_num_accepted, oracle_debug* dbg, int nthreads) {
    if (B < 0 || V <= 0 || !(temperature >= 0.0) || isinf(temperature) || !target || !seq_offsets ||
        !gammas || !out_tokens || !out_num_accepted || nsteps < 1)
        return 1u << OR_ERR_INVALID_ARG;
    if (seq_offsets[0] != 0) return 1u << OR_ERR_BAD_OFFSETS;
    for (int32_t b = 0; b < B; ++b)
        if (gammas[b] < 0 || seq_offsets[b + 1] - seq_offsets[b] != gammas[b]) return 1u << OR_ERR_BAD_OFFSETS;
    if (B == 0) return 0;
    /* draft rows are read only in sampling mode; without them the drafts are point masses */
    if (seq_offsets[B] > 0 && !draft_tokens) return 1u << OR_ERR_INVALID_ARG;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > B) nthreads = B;
    job_t* jobs = (job_t*)calloc((size_t)nthreads, sizeof(job_t));
    pthread_t* th = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
    for (int t = 0; t < nthreads; ++t) {
        job_t* J = &jobs[t];
        J->target = target; J->draft = draft; J->dtype = dtype; J->tok = draft_tokens;
        J->off = seq_offsets; J->gam = gammas; J->B = B; J->V = V; J->T = temperature;
        J->seed = seed; J->step = step; J->out_tok = out_tokens; J->out_n = out_num_accepted;
        J->dbg = dbg;
        J->nsteps = nsteps;
        J->seq_base = seq_base;
        J->b0 = (int32_t)((int64_t)B * t / nthreads);
        J->b1 = (int32_t)((int64_t)B * (t + 1) / nthreads);
    }
    for (int t = 1; t < nthreads; ++t) pthread_create(&th[t], NULL, run_job, &jobs[t]);
    run_job(&jobs[0]);
    uint32_t st = jobs[0].status;
    for (int t = 1; t < nthreads; ++t) {
        pthread_join(th[t], NULL);
        st |= jobs[t].status;
    }
    free(jobs); free(th);
    return st;
}

uint32_t oracle_verify(const void* target, const void* draft, int dtype, const int32_t* draft_tokens,
                       const int32_t* seq_offsets, const int32_t* gammas, int32_t B, int32_t V,
                       double temperature, uint64_t seed, uint64_t step, int32_t* out_tokens,
                       int32_t* out_num_accepted, oracle_debug* dbg, int nthreads) {
    return verify_batch(target, draft, dtype, draft_tokens, seq_offsets, gammas, B, V, temperature, seed, step,
                        0u, 1, out_tokens, out_num_accepted, dbg, nthreads);
}

/*
 * oracle_verify on a contiguous range of a larger batch whose sequence 0 is the batch's sequence
 * seq_base: the uniforms of sequence b are those of the batch's sequence seq_base + b, so verifying the
 * ranges of a batch separately and concatenating their outputs gives the whole batch's outputs.
 */
uint32_t oracle_verify_range(const void* target, const void* draft, int dtype, const int32_t* draft_tokens,
                             const int32_t* seq_offsets, const int32_t* gammas, int32_t B, int32_t V,
                             double temperature, uint64_t seed, uint64_t step, uint32_t seq_base,
                             int32_t* out_tokens, int32_t* out_num_accepted, oracle_debug* dbg, int nthreads) {
    return verify_batch(target, draft, dtype, draft_tokens, seq_offsets, gammas, B, V, temperature, seed, step,
                        seq_base, 1, out_tokens, out_num_accepted, dbg, nthreads);
}

/*
 * oracle_verify for steps step .. step + nsteps - 1 of one batch (sampling mode, temperature > 0): the
 * same rule on the same probabilities, each sequence's softmaxes computed once and its draws made with
 * every step's uniforms. out_tokens [nsteps][R_t] and out_num_accepted [nsteps][B], step-major; debug
 * values of the first step only. Identical to nsteps calls of oracle_verify.
 */
uint32_t oracle_verify_steps(const void* target, const void* draft, int dtype, const int32_t* draft_tokens,
                             const int32_t* seq_offsets, const int32_t* gammas, int32_t B, int32_t V,
                             double temperature, uint64_t seed, uint64_t step, int32_t nsteps,
                             int32_t* out_tokens, int32_t* out_num_accepted, int nthreads) {
    if (!(temperature > 0.0)) return 1u << OR_ERR_INVALID_ARG;
    return verify_batch(target, draft, dtype, draft_tokens, seq_offsets, gammas, B, V, temperature, seed, step,
                        0u, nsteps, out_tokens, out_num_accepted, NULL, nthreads);
}

/*
 * Inverse-CDF bracket of one token for a single draw, used to classify a disagreement as lying
 * inside the decision band. trow/drow point at one target / draft row (drow NULL: draw from p
 * alone, as for the bonus token, or, with x_excl >= 0, from the residual of a point-mass draft at
 * x_excl: p with x_excl removed). Returns the drawn token for uniform u and writes the running
 * sums C_{k-1}/S and C_k/S of token k_query and the normaliser S.
 */
int32_t oracle_draw_bracket(const void* trow, const void* drow, int dtype, int32_t V, double T,
                            double u, int32_t x_excl, int32_t k_query, double* c_lo, double* c_hi,
                            double* S_out) {
    double* p = (double*)malloc(sizeof(double) * (size_t)V);
    double* q = (double*)malloc(sizeof(double) * (size_t)V);
    double* w = (double*)malloc(sizeof(double) * (size_t)V);
    int32_t tok = -1;
    if (row_softmax(trow, dtype, 0, V, T, p, NULL)) goto done;
    double S = 0.0;
    if (drow) {
        if (row_softmax(drow, dtype, 0, V, T, q, NULL)) goto done;
        for (int32_t k = 0; k < V; ++k) { w[k] = p[k] > q[k] ? p[k] - q[k] : 0.0; S += w[k]; }
    } else if (x_excl >= 0 && x_excl < V) { /* point mass at x_excl: max(0, p - q) */
        for (int32_t k = 0; k < V; ++k) { w[k] = k == x_excl ? 0.0 : p[k]; S += w[k]; }
    }
    if ((!drow && !(x_excl >= 0 && x_excl < V)) || S == 0.0) {
        S = 0.0;
        for (int32_t k = 0; k < V; ++k) { w[k] = p[k]; S += w[k]; }
    }
    tok = invcdf(w, V, S, u);
    double c = 0.0;
    for (int32_t k = 0; k < V; ++k) {
        if (k == k_query) *c_lo = c / S;
        c += w[k];
        if (k == k_query) *c_hi = c / S;
    }
    *S_out = S;
done:
    free(p); free(q); free(w);
    return tok;
}

/* ------------------------------------------------------------------------------------------ */
/* Token-tree verification (point-mass candidates)                                            */
/* ------------------------------------------------------------------------------------------ */
/*
 * Reading (the pages sketch tree drafts -- EAGLE's top-K candidates, "Accelerating Sonar through
 * speculation", §"EAGLE" -- but give no rule): the tree's candidates are tokens without a draft
 * distribution, so each is a point mass, and [velog] §2-1/§2-2 is applied to the children of the
 * current node in index order, each rejection removing its token from p:
 *   cur = root; E = {} (removed tokens), P_E = their p mass;
 *   for each child c of cur: x = token[c]; if x in E: rejected;
 *     else accept iff u_c * (1 - P_E) < p_cur(x)   (p restricted to the tokens not removed);
 *     accepted: emit x, cur = c, E = {}; rejected: E += {x}.
 *   No child accepted (or a leaf): draw from p_cur with E removed (E empty: p itself) and stop.
 * The first emitted token is then distributed exactly as p_root. Nodes are numbered 0 (root) ..
 * gamma; node j >= 1 is draft slot j - 1 with parent parents[j - 1] < j. Uniforms: u_c is the accept
 * uniform of slot c - 1, the final draw uses the draw uniform of slot cur -- for a chain (parents[i]
 * = i) this is exactly the linear rule with point-mass drafts.
 */
static int32_t tree_probs(const double* p, const int32_t* parent, const int32_t* x, int32_t gamma, int32_t V,
                          const double* u_acc, const double* u_smp, int32_t* out, int32_t* path) {
    double* w = (double*)malloc(sizeof(double) * (size_t)(V > 0 ? V : 1));
    char* removed = (char*)calloc((size_t)(V > 0 ? V : 1), 1);
    int32_t cur = 0, n = 0;
    for (;;) {
        const double* pc = p + (size_t)cur * V;
        double PE = 0.0;
        int32_t next = -1;
        for (int32_t c = 1; c <= gamma; ++c) {
            if (parent[c - 1] != cur) continue;
            const int32_t xc = x[c - 1];
            if (removed[xc]) continue;
            if (u_acc[c - 1] * (1.0 - PE) < pc[xc]) { next = c; break; }
            removed[xc] = 1;
            PE += pc[xc];
        }
        if (next >= 0) {
            out[n] = x[next - 1];
            if (path) path[n] = next;
            ++n;
            memset(removed, 0, (size_t)V);
            cur = next;
            continue;
        }
        double S = 0.0;
        for (int32_t k = 0; k < V; ++k) { w[k] = removed[k] ? 0.0 : pc[k]; S += w[k]; }
        if (S == 0.0) for (int32_t k = 0; k < V; ++k) { w[k] = pc[k]; S += w[k]; } /* (reading R6) */
        out[n] = invcdf(w, V, S, u_smp[cur]);
        break;
    }
    for (int32_t j = n + 1; j <= gamma; ++j) out[j] = -1;
    if (path) for (int32_t j = n; j < gamma; ++j) path[j] = -1;
    free(w);
    free(removed);
    return n;
}

/* The tree rule on given probabilities (test helper): p [gamma+1, V] (row j: node j), parent/x of the
 * gamma non-root nodes, uniforms by slot. Returns n; out [gamma+1] tokens, path [gamma] nodes. */
int32_t oracle_tree_probs(const double* p, const int32_t* parent, const int32_t* x, int32_t gamma, int32_t V,
                          const double* u_acc, const double* u_smp, int32_t* out, int32_t* path) {
    return tree_probs(p, parent, x, gamma, V, u_acc, u_smp, out, path);
}

/*
 * Verify a batch of token trees: sequence b has gammas[b] + 1 nodes, node j the target row
 * seq_offsets[b] + b + j, non-root node j the draft slot seq_offsets[b] + j - 1 (token draft_tokens[.],
 * parent parents[.] in [0, j)). Outputs as oracle_verify (out_tokens: the accepted path's tokens, then
 * the drawn one) plus out_path [R_d]: the accepted nodes. Greedy (T == 0): the first child whose token
 * is the argmax of the current row is taken; else that argmax is emitted. A bad parent fails the
 * sequence with OR_ERR_BAD_OFFSETS; tokens and non-finite / empty rows as oracle_verify.
 */
uint32_t oracle_verify_tree(const void* target, int dtype, const int32_t* draft_tokens, const int32_t* seq_offsets,
                            const int32_t* gammas, const int32_t* parents, int32_t B, int32_t V, double T,
                            uint64_t seed, uint64_t step, int32_t* out_tokens, int32_t* out_num_accepted,
                            int32_t* out_path) {
    if (B < 0 || V <= 0 || !(T >= 0.0) || isinf(T) || !target || !seq_offsets || !gammas || !out_tokens ||
        !out_num_accepted)
        return 1u << OR_ERR_INVALID_ARG;
    if (seq_offsets[0] != 0) return 1u << OR_ERR_BAD_OFFSETS;
    for (int32_t b = 0; b < B; ++b)
        if (gammas[b] < 0 || seq_offsets[b + 1] - seq_offsets[b] != gammas[b]) return 1u << OR_ERR_BAD_OFFSETS;
    uint32_t status = 0;
    int32_t gmax = 0;
    for (int32_t b = 0; b < B; ++b) gmax = gammas[b] > gmax ? gammas[b] : gmax;
    double* p = (double*)malloc(sizeof(double) * (size_t)V * (size_t)(gmax + 1));
    double* ua = (double*)malloc(sizeof(double) * (size_t)(gmax + 1));
    double* us = (double*)malloc(sizeof(double) * (size_t)(gmax + 1));
    int32_t* arg = (int32_t*)malloc(sizeof(int32_t) * (size_t)(gmax + 1));
    for (int32_t b = 0; b < B; ++b) {
        const int32_t g = gammas[b], d0 = seq_offsets[b], t0 = d0 + b;
        int code = 0;
        for (int32_t i = 0; i < g && !code; ++i) {
            if (draft_tokens[d0 + i] < 0 || draft_tokens[d0 + i] >= V) code = OR_ERR_BAD_TOKEN;
            else if (parents[d0 + i] < 0 || parents[d0 + i] > i) code = OR_ERR_BAD_OFFSETS;
        }
        for (int32_t j = 0; j <= g && !code; ++j)
            code = T == 0.0 ? row_argmax(target, dtype, (size_t)(t0 + j), V, &arg[j])
                            : row_softmax(target, dtype, (size_t)(t0 + j), V, T, p + (size_t)j * V, NULL);
        if (code) {
            for (int32_t j = 0; j <= g; ++j) out_tokens[t0 + j] = -1;
            if (out_path) for (int32_t j = 0; j < g; ++j) out_path[d0 + j] = -1;
            out_num_accepted[b] = -1;
            status |= 1u << code;
            continue;
        }
        int32_t n = 0;
        if (T == 0.0) {
            int32_t cur = 0;
            for (;;) {
                int32_t next = -1;
                for (int32_t c = 1; c <= g && next < 0; ++c)
                    if (parents[d0 + c - 1] == cur && draft_tokens[d0 + c - 1] == arg[cur]) next = c;
                if (next < 0) break;
                out_tokens[t0 + n] = arg[cur];
                if (out_path) out_path[d0 + n] = next;
                ++n;
                cur = next;
            }
            out_tokens[t0 + n] = arg[cur];
            for (int32_t j = n + 1; j <= g; ++j) out_tokens[t0 + j] = -1;
            if (out_path) for (int32_t j = n; j < g; ++j) out_path[d0 + j] = -1;
        } else {
            for (int32_t j = 0; j <= g; ++j) {
                ua[j] = oracle_uniform(seed, step, (uint32_t)b, (uint32_t)j, 0);
                us[j] = oracle_uniform(seed, step, (uint32_t)b, (uint32_t)j, 1);
            }
            n = tree_probs(p, parents + d0, draft_tokens + d0, g, V, ua, us, out_tokens + t0,
                           out_path ? out_path + d0 : NULL);
        }
        out_num_accepted[b] = n;
    }
    free(p); free(ua); free(us); free(arg);
    return status;
}
