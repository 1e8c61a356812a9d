/*
 * spec_oracle.h -- the ORACLE for one hybrid speculative-decoding round.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, __graft_entry__.smoke() and the
 * cpu_baseline / reference legs of bench.py load this library.  The product
 * library (speculative_decoding_draft_spec_gb300) never links, includes or
 * calls it, and it shares no code with the CUDA path.
 *
 * Every function is a plain, slow, single-threaded statement of a definition
 * from the pages:
 *   [HS] "Hybrid Spark: Adaptive Speculative Decoding That Lets the Content
 *        Choose the Drafter" (arXiv 2611.05611v1)
 *   [AS] "AdaSpark: Adaptive DSpark with Online Learning for Tree Verification
 *        and N-gram Fill" (arXiv 2610.05774)
 *   [LS] "Efficient speculative decoding with a fixed-cost parallel drafter"
 *        (LongSpark, arXiv 2609.37029)
 *   [PH] Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as
 *        1, 2, 3", SC'11 (Philox4x32-10)
 *
 * Floating point is double, except where a floating-point value decides an
 * integer result that must match bit for bit (the budget selection): there
 * the pricing values h_k, S_k and V are fp32 with a fixed left-to-right order,
 * the precision the GPU kernel decides in.
 *
 * Return values: a bit mask of ORACLE_ST_* data-error bits (0 = clean), or
 * ORACLE_ERR_ARG (negative) for an unusable argument.
 */
#ifndef SPEC_ORACLE_H
#define SPEC_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ORACLE_ERR_ARG (-1)

/* data-error bits (same meaning as the product's device status word) */
#define ORACLE_ST_BAD_TOKEN  0x1u
#define ORACLE_ST_NONFINITE  0x2u
#define ORACLE_ST_BAD_TREE   0x4u
#define ORACLE_ST_BAD_LENGTH 0x8u
#define ORACLE_ST_BAD_VALUE  0x10u

/* chain-selection policies ([HS] sec. 4.3, sec. 4.5, App. H) */
#define ORACLE_POLICY_PROPOSED    0
#define ORACLE_POLICY_NGRAM_FIRST 1
#define ORACLE_POLICY_EXTENSION   2
#define ORACLE_POLICY_MODEL_ONLY  3
#define ORACLE_POLICY_NGRAM_ONLY  4

/* where the chosen chain came from */
#define ORACLE_SRC_MODEL     0
#define ORACLE_SRC_NGRAM     1
#define ORACLE_SRC_CONTAINS  2
#define ORACLE_SRC_EXTENSION 3

/* Eq. (1) of [HS] sec. 4.2: coefficients of the n-gram acceptance estimator. */
typedef struct {
  double beta[32];               /* beta_k, k = 1..L  (beta[k-1])            */
  double w_first, w_rest;        /* match-length weight, first / later token */
  double delta;                  /* agreement weight                          */
  double ell_first, ell_rest;    /* full-match bonus                          */
  double kappa_first, kappa_rest;/* copy-length weight                        */
  int32_t n_ref;                 /* 5:   (n - n_ref)                          */
  int32_t n_full;                /* 15:  [n = n_full] full-match indicator    */
  int32_t m_cap;                 /* 256: min(m, m_cap)                        */
  int32_t m_ref;                 /* 15:  ln(min(m, m_cap) / m_ref)            */
  int32_t use_constant_h;        /* 1: h_k = constant_h for every k           */
  int32_t pad_;
  double constant_h;
} oracle_estimator;

/* Philox4x32-10 block function [PH]. */
void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2],
                          uint32_t out[4]);
/* the uniform the round uses: (w >> 8) * 2^-24, in [0, 1), exact in fp32 */
double oracle_u01(uint32_t w);
/* u_i (word 0) and u'_i (word 1) for request r, position i (1-based) */
void oracle_round_uniforms(uint64_t seed, uint64_t step, uint32_t r, uint32_t i,
                           double* u, double* u2);

/* A1: n-gram prompt lookup ([HS] sec. 4.1, 4.2 feature list, 5.1). */
int oracle_ngram_propose(const int32_t* hist, int64_t hist_stride,
                         const int32_t* hist_len, int32_t batch,
                         int32_t n_min, int32_t n_max, int32_t max_propose,
                         int32_t copy_cap,
                         int32_t* g, int32_t* g_len, int32_t* match_n,
                         int32_t* agree, int32_t* copy_len);

/* Eq. (1): one acceptance estimate, rounded to fp32. */
float oracle_estimate_h(const oracle_estimator* e, int32_t k, int32_t n,
                        int32_t a, int32_t m);
/* Eq. (3): chain value sum_k max(S_k - lambda, 0), fp32, k order. */
float oracle_chain_value(const float* S, int32_t len, float lambda);

/* A2: pricing, chain choice and batch-wide budget allocation
 * ([HS] Algorithm 1, sec. 4.3, 4.4, 4.5, App. H). */
int oracle_price_and_allocate(
    int32_t batch, int32_t K, int32_t L,
    const int32_t* d, const float* c, const int32_t* d_len,
    const int32_t* g, const int32_t* g_len, const int32_t* match_n,
    const int32_t* agree, const int32_t* copy_len,
    const oracle_estimator* est, float lambda, int32_t budget,
    int32_t max_verify_len, int32_t policy, int32_t draft_greedy,
    int32_t* chain, float* S, int32_t* chain_len, int32_t* source,
    int32_t* verify_len, int32_t* row_off, uint8_t* point_mass);

/* A3: chain verification ([HS] sec. 2, App. H; [LS] verification rule).
 * dtype 0 = fp32, 1 = bf16 (raw uint16 bits).  u_override, when not NULL,
 * gives [batch x (L+1) x 2] uniforms (u_i, u'_i) for i = 1..L+1 instead of
 * Philox.  dbg_* may be NULL.  dbg_pos[r] = the 1-based position whose row
 * was sampled (or whose argmax was emitted), dbg_t[r] = u' * Z and dbg_Z[r] =
 * Z of that draw (normalised probabilities). */
int oracle_verify_chain(
    int32_t batch, int32_t vocab, int32_t dtype,
    const void* target_logits, const int32_t* row_off,
    const void* draft_logits, int32_t K,
    const int32_t* chain, int32_t L, const int32_t* verify_len,
    const uint8_t* point_mass,
    double temperature, uint64_t seed, uint64_t step, const double* u_override,
    int32_t* out_tokens, int32_t* n_accepted, int32_t* n_emitted,
    double* dbg_ratio, double* dbg_u, double* dbg_resid,
    int32_t* dbg_pos, double* dbg_t, double* dbg_Z);

/* The residual distribution r(x) (unnormalised, normalised p and q) that A3
 * samples from for request r at 1-based position i: rejected != 0 gives
 * max(0, p_i - q_i) (or p_i with y_i removed for a point mass), rejected == 0
 * gives p_i itself (the bonus row).  out has vocab entries. */
int oracle_residual_row(
    int32_t vocab, int32_t dtype, const void* target_logits,
    const int32_t* row_off, const void* draft_logits, int32_t K,
    const int32_t* chain, int32_t L, const uint8_t* point_mass,
    double temperature, int32_t r, int32_t i, int32_t rejected, double* out);

/* A4: greedy tree verification ([AS] sec. 2.2, sec. 3.5). */
int oracle_verify_tree(
    int32_t batch, int32_t vocab, int32_t dtype,
    const void* logits, const int32_t* node_off,
    const int32_t* tok, const int32_t* parent, int32_t max_nodes,
    int32_t* path, int32_t* accept_len, int32_t* out_tokens);

/* The candidate tree of one block-drafter round ([AS] sec. 2.2, sec. 3.1
 * Prop. 1, sec. 3.3 Eq. (6), Algorithm 1).  cand_tok / cand_score
 * [batch x P x Kc] (k = 0 the pick), ng_tok [batch x n_chains x Lg] with
 * ng_len[r][c] tokens (chain 0 from the anchor, chain c >= 1 from pick c-1;
 * 1 <= n_chains <= P + 1), ng_score / ng_adj [batch].  Outputs
 * [batch x width]: tok, parent (local, -1 at the anchor), cand_id
 * (candidate index), unused rows -1; n_rows [batch].
 * dbg_Q [batch x (1 + P Kc + n_chains Lg)]: Q per candidate index (-1 past
 * the last), may be NULL. */
int oracle_build_tree(int32_t batch, int32_t P, int32_t Kc, const int32_t* anchor,
                      const int32_t* cand_tok, const float* cand_score,
                      const int32_t* ng_tok, int32_t n_chains, int32_t Lg, const int32_t* ng_len,
                      const float* ng_score, const float* ng_adj, int32_t width,
                      int32_t* tok, int32_t* parent, int32_t* cand_id, int32_t* n_rows,
                      double* dbg_Q);

/* The n-gram chains of a candidate tree ([AS] sec. 2.2, sec. 3.3): chain 0
 * from the anchor (the last token of hist[r][0 .. hist_len[r]-1]) and chain
 * c from pick c-1 (cand_tok[r][c-1][0]), for c = 0..P.  Outputs
 * [batch x (P+1) x Lg]: ng_tok (-1 past the end), ng_ev (evidence: copy
 * length > 0, or minus the follower count); ng_len [batch x (P+1)]. */
int oracle_ngram_fill(const int32_t* hist, int64_t hist_stride, const int32_t* hist_len, int32_t batch,
                      int32_t P, int32_t Kc, const int32_t* cand_tok, int32_t n_min, int32_t copy_cap,
                      int32_t max_depth, int32_t Lg, int32_t* ng_tok, int32_t* ng_len, int32_t* ng_ev);

/* Budget sizing ([HS] sec. 2, sec. 4.3 Eq. (2), sec. 4.4, App. F): over the
 * slots k < min(chain_len[r], max_verify_len) with survivals S [batch x L],
 * b* = the smallest maximiser of G(b) = (batch + sum of the b largest S) /
 * (C0 + p b), lambda = G(b*) p.  G_out (may be NULL) gets G(0..#slots). */
int oracle_size_budget(int32_t batch, int32_t L, const float* S, const int32_t* chain_len,
                       int32_t max_verify_len, double C0, double p, int32_t* b_star,
                       double* lambda, double* G_out);

/* Probabilistic drafting ([HS] sec. 4.5, App. H): y [batch x K], y[r,k-1] =
 * inverse CDF of softmax(z / T) over draft_logits row r K + k - 1 at the
 * uniform of Philox counter (r, 0x40000000 + k, lo32(step), hi32(step)).
 * u_override [batch x K] replaces the uniforms; dbg_u / dbg_q (may be NULL)
 * get the uniform and q of the drawn token. */
int oracle_sample_drafts(int32_t batch, int32_t K, int32_t vocab, int32_t dtype,
                         const void* draft_logits, double temperature, uint64_t seed,
                         uint64_t step, const double* u_override, int32_t* y, double* dbg_u,
                         double* dbg_q);

/* argmax of one row (lowest index on ties); NaN entries are skipped */
int32_t oracle_row_argmax(const void* row, int32_t vocab, int32_t dtype);

#ifdef __cplusplus
}
#endif
#endif
