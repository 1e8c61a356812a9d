/*
 * spec_oracle.c -- the ORACLE: a plain, slow, single-threaded CPU statement of
 * what one hybrid speculative-decoding round computes.
 *
 * TEST INFRASTRUCTURE ONLY (see spec_oracle.h): never linked or called by the
 * product library, and sharing no code with it.  Built with -ffp-contract=off
 * so that every fp32 product and sum below is one correctly rounded operation.
 */
#include "spec_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Philox4x32-10 [PH]: ten rounds of two 32x32->64 multiplies with the       */
/* published multipliers, the key bumped by the published Weyl constants     */
/* between rounds.                                                           */
/* ------------------------------------------------------------------------ */
#define PHILOX_M0 0xD2511F53u
#define PHILOX_M1 0xCD9E8D57u
#define PHILOX_W0 0x9E3779B9u
#define PHILOX_W1 0xBB67AE85u

void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2],
                          uint32_t out[4]) {
  uint32_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
  uint32_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k0 += PHILOX_W0;
      k1 += PHILOX_W1;
    }
    uint64_t prod0 = (uint64_t)PHILOX_M0 * (uint64_t)x0;
    uint64_t prod1 = (uint64_t)PHILOX_M1 * (uint64_t)x2;
    uint32_t hi0 = (uint32_t)(prod0 >> 32), lo0 = (uint32_t)prod0;
    uint32_t hi1 = (uint32_t)(prod1 >> 32), lo1 = (uint32_t)prod1;
    uint32_t y0 = hi1 ^ x1 ^ k0;
    uint32_t y1 = lo1;
    uint32_t y2 = hi0 ^ x3 ^ k1;
    uint32_t y3 = lo0;
    x0 = y0; x1 = y1; x2 = y2; x3 = y3;
  }
  out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

double oracle_u01(uint32_t w) { return (double)(w >> 8) * (1.0 / 16777216.0); }

/* Counter (r, i, lo32(step), hi32(step)), key (lo32(seed), hi32(seed));
 * word 0 is the accept-test uniform u_i, word 1 the draw uniform u'_i. */
void oracle_round_uniforms(uint64_t seed, uint64_t step, uint32_t r, uint32_t i,
                           double* u, double* u2) {
  uint32_t ctr[4] = {r, i, (uint32_t)step, (uint32_t)(step >> 32)};
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t out[4];
  oracle_philox4x32_10(ctr, key, out);
  *u = oracle_u01(out[0]);
  *u2 = oracle_u01(out[1]);
}

/* ------------------------------------------------------------------------ */
/* A1: n-gram prompt lookup.                                                 */
/* [HS] sec. 4.1: the n-gram drafter proposes up to L tokens following the   */
/* longest earlier occurrence of the request's last n_min..n_max tokens;     */
/* sec. 5.1: longest match wins.  Sec. 4.2 defines the features: n the match */
/* length, a = 1 if the runner-up match predicts the same next token or      */
/* there is no runner-up, m how far the match extends backwards (capped).    */
/*                                                                          */
/* Reading: for every earlier end position j (j <= T-2, so a continuation    */
/* token exists) l(j) is the length of the common suffix of x[..j] and       */
/* x[..T-1], capped at copy_cap (and at j+1).  Candidates have l(j) >= n_min;*/
/* they are ranked by (l(j), j) descending: longest copy first, ties to the  */
/* most recent occurrence.  The runner-up is the second candidate in that    */
/* order.  n = min(l, n_max), m = l.  The proposal may run into the suffix.  */
/* ------------------------------------------------------------------------ */
int oracle_ngram_propose(const int32_t* hist, int64_t hist_stride,
                         const int32_t* hist_len, int32_t batch,
                         int32_t n_min, int32_t n_max, int32_t max_propose,
                         int32_t copy_cap,
                         int32_t* g, int32_t* g_len, int32_t* match_n,
                         int32_t* agree, int32_t* copy_len) {
  if (batch < 0 || n_min < 1 || n_max < n_min || max_propose < 0 ||
      copy_cap < n_max || hist_stride < 0)
    return ORACLE_ERR_ARG;
  int status = 0;
  for (int32_t r = 0; r < batch; ++r) {
    for (int32_t i = 0; i < max_propose; ++i) g[(int64_t)r * max_propose + i] = -1;
    g_len[r] = 0;
    match_n[r] = 0;
    agree[r] = 0;
    copy_len[r] = 0;
    const int32_t T = hist_len[r];
    if (T < 0 || (int64_t)T > hist_stride) {
      status |= ORACLE_ST_BAD_LENGTH;
      continue;
    }
    const int32_t* x = hist + (int64_t)r * hist_stride;
    int have_best = 0, have_second = 0;
    int32_t best_l = 0, best_j = 0, second_l = 0, second_j = 0;
    for (int32_t j = 0; j + 1 < T; ++j) {
      int32_t limit = copy_cap < j + 1 ? copy_cap : j + 1;
      int32_t l = 0;
      while (l < limit && x[j - l] == x[T - 1 - l]) ++l;
      if (l < n_min) continue;
      /* rank by (l, j) descending */
      if (!have_best || l > best_l || (l == best_l && j > best_j)) {
        if (have_best) {
          have_second = 1;
          second_l = best_l;
          second_j = best_j;
        }
        have_best = 1;
        best_l = l;
        best_j = j;
      } else if (!have_second || l > second_l || (l == second_l && j > second_j)) {
        have_second = 1;
        second_l = l;
        second_j = j;
      }
    }
    (void)second_l;
    if (!have_best) continue;
    int32_t avail = T - 1 - best_j;
    int32_t len = avail < max_propose ? avail : max_propose;
    for (int32_t i = 0; i < len; ++i)
      g[(int64_t)r * max_propose + i] = x[best_j + 1 + i];
    g_len[r] = len;
    match_n[r] = best_l < n_max ? best_l : n_max;
    agree[r] = (!have_second || x[second_j + 1] == x[best_j + 1]) ? 1 : 0;
    copy_len[r] = best_l;
  }
  return status;
}

/* ------------------------------------------------------------------------ */
/* [HS] sec. 4.2, Eq. (1):                                                   */
/*  h_k = sigma(beta_k + w_pos(k) (n - 5) + delta a                          */
/*              + [n = 15] (ell_pos(k) + kappa_pos(k) ln(min(m, 256) / 15))) */
/* pos(k) separates the first draft position from the later ones.  The      */
/* value is computed in double and rounded once to fp32 (the pricing        */
/* precision).                                                              */
/* ------------------------------------------------------------------------ */
float oracle_estimate_h(const oracle_estimator* e, int32_t k, int32_t n,
                        int32_t a, int32_t m) {
  if (e->use_constant_h) return (float)e->constant_h;
  const int first = (k == 1);
  double z = e->beta[k - 1];
  z = z + (first ? e->w_first : e->w_rest) * (double)(n - e->n_ref);
  z = z + e->delta * (double)a;
  if (n == e->n_full) {
    int32_t mm = m < e->m_cap ? m : e->m_cap;
    double bonus = (first ? e->ell_first : e->ell_rest);
    bonus = bonus + (first ? e->kappa_first : e->kappa_rest) *
                        log((double)mm / (double)e->m_ref);
    z = z + bonus;
  }
  double h = 1.0 / (1.0 + exp(-z));
  return (float)h;
}

/* [HS] sec. 4.3, Eq. (3): V = sum_k max(S_k - lambda, 0), fp32, in k order. */
float oracle_chain_value(const float* S, int32_t len, float lambda) {
  float v = 0.0f;
  for (int32_t k = 0; k < len; ++k) {
    float t = S[k] - lambda;
    if (t > 0.0f) v = v + t;
  }
  return v;
}

typedef struct {
  float s;
  int32_t r, k;
} slot_t;

static int slot_order(const void* pa, const void* pb) {
  const slot_t* a = (const slot_t*)pa;
  const slot_t* b = (const slot_t*)pb;
  if (a->s > b->s) return -1; /* survival descending */
  if (a->s < b->s) return 1;
  if (a->r != b->r) return a->r < b->r ? -1 : 1; /* request ascending */
  if (a->k != b->k) return a->k < b->k ? -1 : 1; /* position ascending */
  return 0;
}

/* ------------------------------------------------------------------------ */
/* A2 ([HS] Algorithm 1; sec. 4.3 chain value, contains rule; sec. 4.4      */
/* allocation into fixed buffers; sec. 4.5 / App. H lossless policies).     */
/*                                                                          */
/* Per request: S^g_k = prod_{j<=k} h_j, S^d_k = prod_{j<=k} c_j (fp32,      */
/* left to right).  PROPOSED: if |g| > |d| and g starts with all of d, keep  */
/* g with S_k = max(S^g_k, S^d_k) for k <= |d| and S_k = S_{k-1} h_k after   */
/* (reading of "then continue with h_k"); else if g matched and V^g >= V^d   */
/* keep g with S^g (ties go to the n-gram chain); else keep d with S^d.      */
/* NGRAM_FIRST: g whenever it matched.  EXTENSION: d unchanged, plus g's     */
/* tail when d is a prefix of g, the tail continuing S from S^d_|d| and      */
/* verified as point masses.  MODEL_ONLY / NGRAM_ONLY: one drafter alone.    */
/*                                                                          */
/* Allocation ([HS] sec. 2 AV): the top-b (request, position) slots by S,    */
/* ties to the lower request then the lower position, over the slots        */
/* k < min(chain_len, max_verify_len).  S never rises along a chain, so each */
/* request keeps a prefix; verify_len is its length and row_off the         */
/* exclusive prefix sum of verify_len + 1 (one extra row per request for the */
/* bonus / correction token).  The slot price lambda acts in the chain      */
/* choice only.                                                             */
/* ------------------------------------------------------------------------ */
int oracle_price_and_allocate(
    int32_t batch, int32_t K, int32_t L,
    const int32_t* d, const float* c, const int32_t* d_len,
    const int32_t* g, const int32_t* g_len, const int32_t* match_n,
    const int32_t* agree, const int32_t* copy_len,
    const oracle_estimator* est, float lambda, int32_t budget,
    int32_t max_verify_len, int32_t policy, int32_t draft_greedy,
    int32_t* chain, float* S, int32_t* chain_len, int32_t* source,
    int32_t* verify_len, int32_t* row_off, uint8_t* point_mass) {
  if (batch < 0 || K < 0 || L < 1 || L > 31 || K > L || budget < 0 ||
      max_verify_len < 0 || policy < 0 || policy > 4)
    return ORACLE_ERR_ARG;
  if (!est->use_constant_h && L > 32) return ORACLE_ERR_ARG;
  int status = 0;
  float* Sg = (float*)malloc(sizeof(float) * (size_t)L);
  float* Sd = (float*)malloc(sizeof(float) * (size_t)L);
  float* h = (float*)malloc(sizeof(float) * (size_t)L);

  for (int32_t r = 0; r < batch; ++r) {
    int32_t* ch = chain + (int64_t)r * L;
    float* Sr = S + (int64_t)r * L;
    uint8_t* pm = point_mass + (int64_t)r * L;
    for (int32_t k = 0; k < L; ++k) {
      ch[k] = -1;
      Sr[k] = 0.0f;
      pm[k] = 0;
    }
    int32_t dl = d_len[r], gl = g_len[r];
    if (dl < 0 || dl > K) {
      status |= ORACLE_ST_BAD_LENGTH;
      dl = dl < 0 ? 0 : K;
    }
    if (gl < 0 || gl > L) {
      status |= ORACLE_ST_BAD_LENGTH;
      gl = gl < 0 ? 0 : L;
    }
    const int32_t* dr = d + (int64_t)r * K;
    const int32_t* gr = g + (int64_t)r * L;

    /* survivals of the n-gram chain, Eq. (1) estimates */
    float run = 1.0f;
    for (int32_t k = 0; k < gl; ++k) {
      h[k] = oracle_estimate_h(est, k + 1, match_n[r], agree[r], copy_len[r]);
      run = run * h[k];
      Sg[k] = run;
    }
    /* survivals of the model chain from its confidences c_k in [0, 1] */
    run = 1.0f;
    for (int32_t k = 0; k < dl; ++k) {
      float ck = c[(int64_t)r * K + k];
      if (!(ck >= 0.0f)) { /* negative or NaN */
        status |= ORACLE_ST_BAD_VALUE;
        ck = 0.0f;
      } else if (ck > 1.0f) {
        status |= ORACLE_ST_BAD_VALUE;
        ck = 1.0f;
      }
      run = run * ck;
      Sd[k] = run;
    }
    /* reading: an empty model chain is contained in nothing */
    int d_prefix_of_g = (dl >= 1 && gl > dl);
    for (int32_t k = 0; d_prefix_of_g && k < dl; ++k)
      if (gr[k] != dr[k]) d_prefix_of_g = 0;

    int src = ORACLE_SRC_MODEL;
    switch (policy) {
      case ORACLE_POLICY_PROPOSED:
        if (d_prefix_of_g)
          src = ORACLE_SRC_CONTAINS;
        else if (gl > 0 && oracle_chain_value(Sg, gl, lambda) >=
                               oracle_chain_value(Sd, dl, lambda))
          src = ORACLE_SRC_NGRAM;
        else
          src = ORACLE_SRC_MODEL;
        break;
      case ORACLE_POLICY_NGRAM_FIRST:
        src = gl > 0 ? ORACLE_SRC_NGRAM : ORACLE_SRC_MODEL;
        break;
      case ORACLE_POLICY_EXTENSION:
        src = d_prefix_of_g ? ORACLE_SRC_EXTENSION : ORACLE_SRC_MODEL;
        break;
      case ORACLE_POLICY_MODEL_ONLY:
        src = ORACLE_SRC_MODEL;
        break;
      case ORACLE_POLICY_NGRAM_ONLY:
        src = ORACLE_SRC_NGRAM;
        break;
    }
    int32_t len = 0;
    if (src == ORACLE_SRC_MODEL) {
      len = dl;
      for (int32_t k = 0; k < dl; ++k) {
        ch[k] = dr[k];
        Sr[k] = Sd[k];
        pm[k] = draft_greedy ? 1 : 0;
      }
    } else if (src == ORACLE_SRC_NGRAM) {
      len = gl;
      for (int32_t k = 0; k < gl; ++k) {
        ch[k] = gr[k];
        Sr[k] = Sg[k];
        pm[k] = 1;
      }
    } else if (src == ORACLE_SRC_CONTAINS) {
      len = gl;
      float prev = 1.0f;
      for (int32_t k = 0; k < gl; ++k) {
        ch[k] = gr[k];
        if (k < dl)
          Sr[k] = Sg[k] > Sd[k] ? Sg[k] : Sd[k];
        else
          Sr[k] = prev * h[k];
        prev = Sr[k];
        pm[k] = 1;
      }
    } else { /* EXTENSION */
      len = gl;
      float prev = 1.0f;
      for (int32_t k = 0; k < gl; ++k) {
        ch[k] = gr[k]; /* equals d for k < dl */
        if (k < dl) {
          Sr[k] = Sd[k];
          pm[k] = draft_greedy ? 1 : 0;
        } else {
          Sr[k] = prev * h[k];
          pm[k] = 1;
        }
        prev = Sr[k];
      }
    }
    chain_len[r] = len;
    source[r] = src;
  }

  /* batch-wide allocation: top-b slots by (S desc, r asc, k asc) */
  int64_t nslots = 0;
  for (int32_t r = 0; r < batch; ++r) {
    int32_t lim = chain_len[r] < max_verify_len ? chain_len[r] : max_verify_len;
    nslots += lim;
  }
  slot_t* slots = (slot_t*)malloc(sizeof(slot_t) * (size_t)(nslots > 0 ? nslots : 1));
  int64_t ns = 0;
  for (int32_t r = 0; r < batch; ++r) {
    int32_t lim = chain_len[r] < max_verify_len ? chain_len[r] : max_verify_len;
    for (int32_t k = 0; k < lim; ++k) {
      slots[ns].s = S[(int64_t)r * L + k];
      slots[ns].r = r;
      slots[ns].k = k;
      ++ns;
    }
  }
  qsort(slots, (size_t)ns, sizeof(slot_t), slot_order);
  int64_t take = budget < ns ? budget : ns;
  for (int32_t r = 0; r < batch; ++r) verify_len[r] = 0;
  for (int64_t t = 0; t < take; ++t) verify_len[slots[t].r] += 1;
  row_off[0] = 0;
  for (int32_t r = 0; r < batch; ++r) row_off[r + 1] = row_off[r] + verify_len[r] + 1;

  free(slots);
  free(Sg);
  free(Sd);
  free(h);
  return status;
}

/* ------------------------------------------------------------------------ */
/* Rows of logits.                                                           */
/* ------------------------------------------------------------------------ */
static double logit_at(const void* base, int64_t idx, int32_t dtype) {
  if (dtype == 0) return (double)((const float*)base)[idx];
  uint32_t bits = (uint32_t)((const uint16_t*)base)[idx] << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* 1 if the row holds a NaN or +Inf (-Inf is a legal mask value) */
static int row_nonfinite(const void* base, int64_t row, int32_t vocab, int32_t dtype) {
  for (int32_t x = 0; x < vocab; ++x) {
    double z = logit_at(base, row * vocab + x, dtype);
    if (z != z || z == INFINITY) return 1;
  }
  return 0;
}

/* argmax with the lowest index on ties; NaN entries never win. */
static int32_t row_argmax(const void* base, int64_t row, int32_t vocab, int32_t dtype) {
  int32_t best = -1;
  double bv = 0.0;
  for (int32_t x = 0; x < vocab; ++x) {
    double z = logit_at(base, row * vocab + x, dtype);
    if (z != z) continue;
    if (best < 0 || z > bv) {
      best = x;
      bv = z;
    }
  }
  return best < 0 ? 0 : best;
}

int32_t oracle_row_argmax(const void* row, int32_t vocab, int32_t dtype) {
  return row_argmax(row, 0, vocab, dtype);
}

/* softmax(z / T) of one row in double, max-subtracted */
static void row_softmax(const void* base, int64_t row, int32_t vocab, int32_t dtype,
                        double T, double* p) {
  double m = -INFINITY;
  for (int32_t x = 0; x < vocab; ++x) {
    double z = logit_at(base, row * vocab + x, dtype);
    if (z > m) m = z;
  }
  double s = 0.0;
  for (int32_t x = 0; x < vocab; ++x) {
    p[x] = exp((logit_at(base, row * vocab + x, dtype) - m) / T);
    s += p[x];
  }
  for (int32_t x = 0; x < vocab; ++x) p[x] /= s;
}

/* inverse CDF in vocabulary order: the smallest x whose running sum exceeds
 * t; when rounding leaves t at or above the total, the last x with mass. */
static int32_t inverse_cdf(const double* w, int32_t vocab, double t) {
  double run = 0.0;
  int32_t last = 0;
  for (int32_t x = 0; x < vocab; ++x) {
    if (w[x] > 0.0) last = x;
    run += w[x];
    if (run > t) return x;
  }
  return last;
}

/* residual r(x) for a rejected draft y: max(0, p - q), or p with y removed
 * for a point mass (q = delta_y).  Falls back to p when the residual mass is
 * below 1e-30 (reading: an exactly-zero residual has no distribution). */
static double build_residual(const double* p, const double* q, int32_t y,
                             int32_t vocab, int pm, double* out) {
  double Z = 0.0;
  for (int32_t x = 0; x < vocab; ++x) {
    double v;
    if (pm)
      v = (x == y) ? 0.0 : p[x];
    else
      v = p[x] - q[x] > 0.0 ? p[x] - q[x] : 0.0;
    out[x] = v;
    Z += v;
  }
  if (Z <= 1e-30) {
    Z = 0.0;
    for (int32_t x = 0; x < vocab; ++x) {
      out[x] = p[x];
      Z += p[x];
    }
  }
  return Z;
}

/* ------------------------------------------------------------------------ */
/* A3: chain verification.                                                   */
/* [HS] sec. 2: the target scores the draft chain in one pass and accepts    */
/* the longest prefix that passes rejection sampling, plus one token of its  */
/* own; App. H: greedy drafts are verified as point masses.  [LS]: accept y_i*/
/* with probability min(1, p_i(y_i) / q_i(y_i)); at the first rejection      */
/* sample a correction from norm(max(0, p_i - q_i)); if all B candidates are */
/* accepted sample a bonus from p_{B+1}; r accepted => r + 1 tokens.         */
/* T = 0 (greedy target): accept iff y_i = argmax z_i, emit argmax.          */
/* Row i-1 of a request (row_off[r] + i - 1) holds the logits z_i of         */
/* position i; row verify_len holds the bonus position.                      */
/* ------------------------------------------------------------------------ */
int oracle_verify_chain(
    int32_t batch, int32_t vocab, int32_t dtype,
    const void* target_logits, const int32_t* row_off,
    const void* draft_logits, int32_t K,
    const int32_t* chain, int32_t L, const int32_t* verify_len,
    const uint8_t* point_mass,
    double temperature, uint64_t seed, uint64_t step, const double* u_override,
    int32_t* out_tokens, int32_t* n_accepted, int32_t* n_emitted,
    double* dbg_ratio, double* dbg_u, double* dbg_resid,
    int32_t* dbg_pos, double* dbg_t, double* dbg_Z) {
  if (batch < 0 || vocab < 1 || (dtype != 0 && dtype != 1) || L < 1 || L > 31 ||
      K < 0 || !(temperature == temperature))
    return ORACLE_ERR_ARG;
  int status = 0;
  const int greedy = !(temperature > 0.0);
  double* p = (double*)malloc(sizeof(double) * (size_t)vocab);
  double* q = (double*)malloc(sizeof(double) * (size_t)vocab);
  double* w = (double*)malloc(sizeof(double) * (size_t)vocab);
  const int32_t total_rows = row_off[batch];

  for (int32_t r = 0; r < batch; ++r) {
    int32_t* out = out_tokens + (int64_t)r * (L + 1);
    for (int32_t j = 0; j <= L; ++j) out[j] = -1;
    n_accepted[r] = 0;
    n_emitted[r] = 0;
    for (int32_t j = 0; j < L; ++j) {
      if (dbg_ratio) dbg_ratio[(int64_t)r * L + j] = -1.0;
      if (dbg_u) dbg_u[(int64_t)r * L + j] = -1.0;
    }
    if (dbg_resid) dbg_resid[r] = -1.0;
    if (dbg_pos) dbg_pos[r] = 0;
    if (dbg_t) dbg_t[r] = 0.0;
    if (dbg_Z) dbg_Z[r] = 0.0;

    const int32_t ell = verify_len[r];
    const int32_t base = row_off[r];
    if (ell < 0 || ell > L || base < 0 || (int64_t)base + ell >= row_off[r + 1] ||
        row_off[r + 1] > total_rows) {
      status |= ORACLE_ST_BAD_LENGTH;
      continue;
    }
    const int32_t* y = chain + (int64_t)r * L;
    /* which positions carry a draft distribution q (the rest are point masses) */
    int use_q[32];
    for (int32_t i = 1; i <= ell; ++i) {
      int pm = point_mass ? (point_mass[(int64_t)r * L + i - 1] != 0) : 1;
      if (!pm && (greedy || draft_logits == NULL)) pm = 1;
      if (!pm && i > K) {
        status |= ORACLE_ST_BAD_LENGTH;
        pm = 1;
      }
      use_q[i] = !pm;
    }
    /* non-finite scan over every row the request's verification covers */
    for (int32_t i = 0; i <= ell; ++i)
      if (row_nonfinite(target_logits, (int64_t)base + i, vocab, dtype))
        status |= ORACLE_ST_NONFINITE;
    for (int32_t i = 1; i <= ell; ++i)
      if (use_q[i] && row_nonfinite(draft_logits, (int64_t)r * K + i - 1, vocab, dtype))
        status |= ORACLE_ST_NONFINITE;
    for (int32_t i = 1; i <= ell; ++i)
      if (y[i - 1] < 0 || y[i - 1] >= vocab) status |= ORACLE_ST_BAD_TOKEN;

    int32_t acc = 0;
    int rejected = 0;
    if (greedy) {
      for (int32_t i = 1; i <= ell; ++i) {
        int32_t a = row_argmax(target_logits, (int64_t)base + i - 1, vocab, dtype);
        int ok = (y[i - 1] == a);
        if (dbg_ratio) dbg_ratio[(int64_t)r * L + i - 1] = ok ? 1.0 : 0.0;
        if (dbg_u) dbg_u[(int64_t)r * L + i - 1] = 0.0;
        if (ok) {
          out[i - 1] = y[i - 1];
          ++acc;
        } else {
          out[i - 1] = a;
          rejected = 1;
          if (dbg_pos) dbg_pos[r] = i;
          break;
        }
      }
      if (!rejected) {
        out[ell] = row_argmax(target_logits, (int64_t)base + ell, vocab, dtype);
        if (dbg_pos) dbg_pos[r] = ell + 1;
      }
      if (dbg_resid) dbg_resid[r] = 1.0;
    } else {
      for (int32_t i = 1; i <= ell && !rejected; ++i) {
        double u, u2;
        if (u_override) {
          u = u_override[((int64_t)r * (L + 1) + (i - 1)) * 2 + 0];
          u2 = u_override[((int64_t)r * (L + 1) + (i - 1)) * 2 + 1];
        } else {
          oracle_round_uniforms(seed, step, (uint32_t)r, (uint32_t)i, &u, &u2);
        }
        row_softmax(target_logits, (int64_t)base + i - 1, vocab, dtype, temperature, p);
        if (use_q[i])
          row_softmax(draft_logits, (int64_t)r * K + i - 1, vocab, dtype, temperature, q);
        const int32_t yi = y[i - 1];
        const int valid = (yi >= 0 && yi < vocab);
        double ratio;
        if (!valid)
          ratio = 0.0;
        else if (!use_q[i])
          ratio = p[yi];
        else
          ratio = p[yi] / q[yi];
        if (dbg_ratio) dbg_ratio[(int64_t)r * L + i - 1] = ratio;
        if (dbg_u) dbg_u[(int64_t)r * L + i - 1] = u;
        int accept = (ratio >= 1.0) || (u < ratio);
        if (accept) {
          out[i - 1] = yi;
          ++acc;
          continue;
        }
        rejected = 1;
        double Z = build_residual(p, use_q[i] ? q : NULL, valid ? yi : -1, vocab,
                                  !use_q[i], w);
        double t = u2 * Z;
        int32_t xs = inverse_cdf(w, vocab, t);
        out[i - 1] = xs;
        if (dbg_resid) dbg_resid[r] = w[xs] / Z;
        if (dbg_pos) dbg_pos[r] = i;
        if (dbg_t) dbg_t[r] = t;
        if (dbg_Z) dbg_Z[r] = Z;
      }
      if (!rejected) {
        double u, u2;
        if (u_override) {
          u = u_override[((int64_t)r * (L + 1) + ell) * 2 + 0];
          u2 = u_override[((int64_t)r * (L + 1) + ell) * 2 + 1];
        } else {
          oracle_round_uniforms(seed, step, (uint32_t)r, (uint32_t)(ell + 1), &u, &u2);
        }
        (void)u;
        row_softmax(target_logits, (int64_t)base + ell, vocab, dtype, temperature, p);
        double Z = 0.0;
        for (int32_t x = 0; x < vocab; ++x) Z += p[x];
        double t = u2 * Z;
        int32_t xs = inverse_cdf(p, vocab, t);
        out[ell] = xs;
        if (dbg_resid) dbg_resid[r] = p[xs] / Z;
        if (dbg_pos) dbg_pos[r] = ell + 1;
        if (dbg_t) dbg_t[r] = t;
        if (dbg_Z) dbg_Z[r] = Z;
      }
    }
    n_accepted[r] = acc;
    n_emitted[r] = acc + 1;
  }
  free(p);
  free(q);
  free(w);
  return status;
}

int oracle_residual_row(
    int32_t vocab, int32_t dtype, const void* target_logits,
    const int32_t* row_off, const void* draft_logits, int32_t K,
    const int32_t* chain, int32_t L, const uint8_t* point_mass,
    double temperature, int32_t r, int32_t i, int32_t rejected, double* out) {
  if (vocab < 1 || !(temperature > 0.0) || i < 1) return ORACLE_ERR_ARG;
  double* p = (double*)malloc(sizeof(double) * (size_t)vocab);
  double* q = (double*)malloc(sizeof(double) * (size_t)vocab);
  row_softmax(target_logits, (int64_t)row_off[r] + i - 1, vocab, dtype, temperature, p);
  if (!rejected) {
    for (int32_t x = 0; x < vocab; ++x) out[x] = p[x];
  } else {
    int pm = point_mass ? (point_mass[(int64_t)r * L + i - 1] != 0) : 1;
    if (!pm && (draft_logits == NULL || i > K)) pm = 1;
    if (!pm) row_softmax(draft_logits, (int64_t)r * K + i - 1, vocab, dtype, temperature, q);
    int32_t yi = chain[(int64_t)r * L + i - 1];
    int valid = (yi >= 0 && yi < vocab);
    build_residual(p, pm ? NULL : q, valid ? yi : -1, vocab, pm, out);
  }
  free(p);
  free(q);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* A4: greedy tree verification ([AS] sec. 2.2).  A candidate is accepted   */
/* when its token equals the target's argmax at its parent's row and its    */
/* parent is accepted; at most one child of an accepted node can match, so  */
/* the accepted nodes form one path from the anchor; the round commits that */
/* path and the argmax at its last node.  Reading for duplicate sibling     */
/* tokens: the lowest-index child wins.                                     */
/* Node 0 of each request is the anchor (parent -1); parents precede their  */
/* children.                                                                */
/* ------------------------------------------------------------------------ */
int oracle_verify_tree(
    int32_t batch, int32_t vocab, int32_t dtype,
    const void* logits, const int32_t* node_off,
    const int32_t* tok, const int32_t* parent, int32_t max_nodes,
    int32_t* path, int32_t* accept_len, int32_t* out_tokens) {
  if (batch < 0 || vocab < 1 || (dtype != 0 && dtype != 1) || max_nodes < 1)
    return ORACLE_ERR_ARG;
  int status = 0;
  for (int32_t r = 0; r < batch; ++r) {
    for (int32_t j = 0; j < max_nodes; ++j) {
      path[(int64_t)r * max_nodes + j] = -1;
      out_tokens[(int64_t)r * max_nodes + j] = -1;
    }
    accept_len[r] = -1;
    const int32_t base = node_off[r];
    const int32_t n = node_off[r + 1] - base;
    if (base < 0 || n < 1 || n > max_nodes || node_off[r + 1] > node_off[batch]) {
      status |= ORACLE_ST_BAD_LENGTH;
      continue;
    }
    int ok = (parent[base] == -1);
    for (int32_t j = 1; j < n; ++j)
      if (parent[base + j] < 0 || parent[base + j] >= j) ok = 0;
    if (!ok) {
      status |= ORACLE_ST_BAD_TREE;
      continue;
    }
    for (int32_t j = 1; j < n; ++j)
      if (tok[base + j] < 0 || tok[base + j] >= vocab) status |= ORACLE_ST_BAD_TOKEN;
    for (int32_t j = 0; j < n; ++j)
      if (row_nonfinite(logits, (int64_t)base + j, vocab, dtype)) status |= ORACLE_ST_NONFINITE;

    int32_t cur = 0, len = 1;
    path[(int64_t)r * max_nodes] = 0;
    int32_t a = row_argmax(logits, (int64_t)base, vocab, dtype);
    for (;;) {
      int32_t next = -1;
      for (int32_t ch = cur + 1; ch < n; ++ch)
        if (parent[base + ch] == cur && tok[base + ch] == a) {
          next = ch;
          break;
        }
      if (next < 0) break;
      out_tokens[(int64_t)r * max_nodes + len - 1] = tok[base + next];
      path[(int64_t)r * max_nodes + len] = next;
      ++len;
      cur = next;
      a = row_argmax(logits, (int64_t)base + cur, vocab, dtype);
    }
    out_tokens[(int64_t)r * max_nodes + len - 1] = a;
    accept_len[r] = len - 1;
  }
  return status;
}

/* ------------------------------------------------------------------------ */
/* The candidate tree of one block-drafter round ([AS] sec. 2.2 tree shape; */
/* sec. 3.3 n-gram candidates and Eq. (6); sec. 3.1, Prop. 1, best-first    */
/* order; Algorithm 1: the first n-1 nodes, laid out depth-first).          */
/*                                                                          */
/* Candidates: 0 the anchor; 1 + i Kc + k the k-th ranked candidate of      */
/* block position i (k = 0 the pick, k >= 1 its siblings); the picks form a */
/* spine (pick i under pick i-1, pick 0 under the anchor) and the siblings  */
/* of position i hang from the pick's parent as leaves.  n-gram chains: c = */
/* 0 starts at the anchor, c >= 1 at pick c-1 (the chains branch from the   */
/* anchor and from each pick), taken in order c = 0, 1, ...  A step whose   */
/* token equals a drafter child of the current node marks that child agreed */
/* and moves to it (the lowest index on duplicates); else, when an n-gram   */
/* node with that token already hangs from the current node (an earlier     */
/* chain's), it moves to it; else it appends an n-gram node under the       */
/* current node and moves to it.  At every node a chain passes through, the */
/* drafter children other than the one it moves to are contradicted.       */
/* Reading: a candidate that one chain agrees with and another contradicts  */
/* counts as agreed.                                                        */
/* Scores: a drafter candidate keeps its given s, plus adj if agreed, minus */
/* adj if contradicted (adj = max(0, logit p_src) from the caller; reading: */
/* the agreed / contradiction bucket weights are zero, their prior); an     */
/* n-gram node scores ng_score.  Scores are clamped to [-80, 80].           */
/* q_j = exp(s_j) / (1 + sum over the children c of parent(j) of exp(s_c))  */
/* (children summed in index order); Q_j = Q_parent(j) q_j, Q_0 = 1.  The   */
/* order is Q descending, ties to the lower index; the tree is the anchor   */
/* and the first width-1 candidates of the order, laid out depth-first with */
/* children in increasing candidate index (reading: the page fixes no child */
/* order).  All in double.                                                  */
/* ------------------------------------------------------------------------ */
int oracle_build_tree(int32_t batch, int32_t P, int32_t Kc, const int32_t* anchor,
                      const int32_t* cand_tok, const float* cand_score,
                      const int32_t* ng_tok, int32_t n_chains, int32_t Lg, const int32_t* ng_len,
                      const float* ng_score, const float* ng_adj, int32_t width,
                      int32_t* tok, int32_t* parent, int32_t* cand_id, int32_t* n_rows,
                      double* dbg_Q) {
  if (batch < 0 || P < 0 || Kc < 1 || Lg < 0 || width < 1 || n_chains < 1 || n_chains > P + 1)
    return ORACLE_ERR_ARG;
  const int32_t cap = 1 + P * Kc + n_chains * Lg;
  int32_t* ctok = (int32_t*)malloc(sizeof(int32_t) * (size_t)cap);
  int32_t* cpar = (int32_t*)malloc(sizeof(int32_t) * (size_t)cap);
  int32_t* drafter = (int32_t*)malloc(sizeof(int32_t) * (size_t)cap);
  int32_t* agreed = (int32_t*)malloc(sizeof(int32_t) * (size_t)cap);
  int32_t* contra = (int32_t*)malloc(sizeof(int32_t) * (size_t)cap);
  int32_t* chosen = (int32_t*)malloc(sizeof(int32_t) * (size_t)cap);
  int32_t* order = (int32_t*)malloc(sizeof(int32_t) * (size_t)cap);
  int32_t* pos = (int32_t*)malloc(sizeof(int32_t) * (size_t)cap);
  double* s = (double*)malloc(sizeof(double) * (size_t)cap);
  double* q = (double*)malloc(sizeof(double) * (size_t)cap);
  double* Q = (double*)malloc(sizeof(double) * (size_t)cap);
  int status = 0;
  for (int32_t r = 0; r < batch; ++r) {
    /* the drafter's block */
    int32_t N = 1 + P * Kc;
    ctok[0] = anchor[r];
    cpar[0] = -1;
    drafter[0] = 0;
    agreed[0] = contra[0] = 0;
    s[0] = 0.0;
    for (int32_t i = 0; i < P; ++i)
      for (int32_t k = 0; k < Kc; ++k) {
        const int32_t j = 1 + i * Kc + k;
        ctok[j] = cand_tok[((int64_t)r * P + i) * Kc + k];
        cpar[j] = (i == 0) ? 0 : 1 + (i - 1) * Kc;
        drafter[j] = 1;
        agreed[j] = contra[j] = 0;
        s[j] = (double)cand_score[((int64_t)r * P + i) * Kc + k];
      }
    /* the n-gram chains, from the anchor (c = 0) and from pick c - 1 */
    for (int32_t ch = 0; ch < n_chains; ++ch) {
      int32_t gl = ng_len[(int64_t)r * n_chains + ch];
      if (gl < 0 || gl > Lg) {
        status |= ORACLE_ST_BAD_LENGTH;
        gl = 0;
      }
      int32_t cur = (ch == 0) ? 0 : 1 + (ch - 1) * Kc;
      for (int32_t t = 0; t < gl; ++t) {
        const int32_t x = ng_tok[((int64_t)r * n_chains + ch) * Lg + t];
        int32_t hit = -1;
        for (int32_t c = cur + 1; c < N; ++c)
          if (drafter[c] && cpar[c] == cur && ctok[c] == x) {
            hit = c;
            break;
          }
        for (int32_t c = cur + 1; c < N; ++c)
          if (drafter[c] && cpar[c] == cur && c != hit) contra[c] = 1;
        if (hit >= 0) {
          agreed[hit] = 1;
          cur = hit;
          continue;
        }
        int32_t old = -1;
        for (int32_t c = 1 + P * Kc; c < N; ++c)
          if (cpar[c] == cur && ctok[c] == x) {
            old = c;
            break;
          }
        if (old >= 0) {
          cur = old;
          continue;
        }
        ctok[N] = x;
        cpar[N] = cur;
        drafter[N] = 0;
        agreed[N] = contra[N] = 0;
        s[N] = (double)ng_score[r];
        cur = N;
        ++N;
      }
    }
    const double adj = (double)ng_adj[r];
    for (int32_t j = 1; j < N; ++j) {
      if (drafter[j]) s[j] += agreed[j] ? adj : (contra[j] ? -adj : 0.0);
      if (s[j] > 80.0) s[j] = 80.0;
      if (s[j] < -80.0) s[j] = -80.0;
    }
    /* Eq. (6): one softmax per parent over its children and "none" */
    for (int32_t p = 0; p < N; ++p) {
      double den = 1.0;
      for (int32_t c = p + 1; c < N; ++c)
        if (cpar[c] == p) den += exp(s[c]);
      for (int32_t c = p + 1; c < N; ++c)
        if (cpar[c] == p) q[c] = exp(s[c]) / den;
    }
    Q[0] = 1.0;
    for (int32_t j = 1; j < N; ++j) Q[j] = Q[cpar[j]] * q[j];
    if (dbg_Q) {
      for (int32_t j = 0; j < cap; ++j) dbg_Q[(int64_t)r * cap + j] = j < N ? Q[j] : -1.0;
    }
    /* best-first order (insertion sort: Q descending, ties to the lower index) */
    int32_t m = 0;
    for (int32_t j = 1; j < N; ++j) {
      int32_t at = m;
      while (at > 0 && (Q[order[at - 1]] < Q[j])) --at;
      for (int32_t z = m; z > at; --z) order[z] = order[z - 1];
      order[at] = j;
      ++m;
    }
    const int32_t take = (width - 1 < m) ? width - 1 : m;
    for (int32_t j = 0; j < N; ++j) chosen[j] = (j == 0);
    for (int32_t z = 0; z < take; ++z) chosen[order[z]] = 1;
    /* depth-first layout, children in increasing candidate index */
    int32_t n = 0;
    int32_t* stack = order; /* reuse: the order is no longer needed */
    int32_t sp = 0;
    stack[sp++] = 0;
    while (sp > 0) {
      const int32_t j = stack[--sp];
      pos[j] = n;
      tok[(int64_t)r * width + n] = ctok[j];
      parent[(int64_t)r * width + n] = (j == 0) ? -1 : pos[cpar[j]];
      cand_id[(int64_t)r * width + n] = j;
      ++n;
      for (int32_t c = N - 1; c > j; --c) /* pushed in decreasing index: popped increasing */
        if (chosen[c] && cpar[c] == j) stack[sp++] = c;
    }
    for (int32_t z = n; z < width; ++z) {
      tok[(int64_t)r * width + z] = -1;
      parent[(int64_t)r * width + z] = -1;
      cand_id[(int64_t)r * width + z] = -1;
    }
    n_rows[r] = n;
  }
  free(ctok);
  free(cpar);
  free(drafter);
  free(agreed);
  free(contra);
  free(chosen);
  free(order);
  free(pos);
  free(s);
  free(q);
  free(Q);
  return status;
}

/* ------------------------------------------------------------------------ */
/* N-gram fill of the candidate tree ([AS] sec. 2.2: chains branch from the */
/* anchor and from each pick and may run past the drafter's block; sec. 3.3 */
/* "N-gram candidates"; the parameter table: last 3 tokens, depth 32).      */
/*                                                                          */
/* x = hist[r][0 .. T-1] is the request's committed text, ending with the   */
/* anchor.  Chain c = 0 starts at the anchor (depth 0), chain c >= 1 at     */
/* pick c-1 (depth c), with context ctx = x, pick_0, ..., pick_{c-1}.  Each */
/* step appends one token y to the chain and to ctx:                        */
/*  1. when the chain is reading along an earlier passage of x and the      */
/*     passage continues (its next position is <= T-1), y is that token;   */
/*  2. else the earlier occurrence of the current context: for every end    */
/*     position j <= T-2 of x, l(j) = common-suffix length of x[..j] and    */
/*     ctx, capped at copy_cap and j+1; candidates have l >= n_min, ranked  */
/*     by (l, j) descending (the n-gram lookup's ranking); y = x[j+1] of    */
/*     the best, and the chain reads on along x from j+2;                   */
/*  3. else the most frequent follower of the last three tokens of ctx:     */
/*     over j in [2, T-2] with x[j-2..j] equal to them, y = the follower    */
/*     x[j+1] with the most occurrences, ties to the follower whose latest  */
/*     occurrence is the most recent; the next step looks up again;         */
/*  4. else the chain stops (nothing is proposed).                          */
/* A chain stops at depth max_depth below the anchor (at most Lg tokens).   */
/* ev: the evidence of each token: the length of the copy it continues (the */
/* lookup's l, plus one per token read since, capped at copy_cap) for steps */
/* 1-2, minus the follower's count for step 3.                              */
/* Readings: "an earlier occurrence of the current context" takes the      */
/* n-gram lookup's ranking with its minimum n_min (so step 3 can fire only  */
/* when n_min > 3); a passage is read only within x.                        */
/* ------------------------------------------------------------------------ */
int oracle_ngram_fill(const int32_t* hist, int64_t hist_stride, const int32_t* hist_len, int32_t batch,
                      int32_t P, int32_t Kc, const int32_t* cand_tok, int32_t n_min, int32_t copy_cap,
                      int32_t max_depth, int32_t Lg, int32_t* ng_tok, int32_t* ng_len, int32_t* ng_ev) {
  if (batch < 0 || P < 0 || Kc < 1 || n_min < 1 || copy_cap < n_min || max_depth < 0 || Lg < 0 ||
      hist_stride < 0)
    return ORACLE_ERR_ARG;
  int status = 0;
  const int32_t C = P + 1;
  int32_t* ext = (int32_t*)malloc(sizeof(int32_t) * (size_t)(P + Lg + 1));
  for (int32_t r = 0; r < batch; ++r) {
    const int32_t* x = hist + (int64_t)r * hist_stride;
    int32_t T = hist_len[r];
    if (T < 0 || T > hist_stride) {
      status |= ORACLE_ST_BAD_LENGTH;
      T = 0;
    }
    for (int32_t c = 0; c < C; ++c) {
      int32_t* out = ng_tok + ((int64_t)r * C + c) * Lg;
      int32_t* ev = ng_ev + ((int64_t)r * C + c) * Lg;
      for (int32_t k = 0; k < Lg; ++k) {
        out[k] = -1;
        ev[k] = 0;
      }
      int32_t cap = max_depth - c;
      if (cap > Lg) cap = Lg;
      int32_t n = 0;
      /* ctx = x ++ ext[0 .. m-1]: the picks on the path, then the chain */
      int32_t m = 0;
      for (int32_t i = 0; i < c; ++i) ext[m++] = cand_tok[((int64_t)r * P + i) * Kc];
      if (T < 1) cap = 0; /* no anchor */
      int64_t q = -1;     /* the passage's next position in x, or -1 */
      int32_t run = 0;    /* the length of the copy being continued */
      while (n < cap) {
        const int64_t len = (int64_t)T + m;
#define CTX(i) ((i) < T ? x[(i)] : ext[(i) - T])
        int32_t y = -1, e = 0, found = 0;
        if (q >= 0 && q <= T - 1) {
          found = 1;
          y = x[q];
          ++q;
          ++run;
          if (run > copy_cap) run = copy_cap;
          e = run;
        } else {
          int32_t top_l = 0;
          int64_t top_j = -1;
          for (int64_t j = 0; j <= (int64_t)T - 2; ++j) {
            int32_t l = 0;
            while (l < copy_cap && l <= j && x[j - l] == CTX(len - 1 - l)) ++l;
            if (l >= n_min && (l > top_l || (l == top_l && j > top_j))) {
              top_l = l;
              top_j = j;
            }
          }
          if (top_j >= 0) {
            found = 1;
            y = x[top_j + 1];
            q = top_j + 2;
            run = top_l;
            e = run;
          } else if (len >= 3) {
            /* followers of the last three tokens: counts and latest positions */
            const int32_t a = CTX(len - 3), b = CTX(len - 2), d = CTX(len - 1);
            int32_t best_cnt = 0;
            int64_t best_last = -1;
            for (int64_t j = 2; j <= (int64_t)T - 2; ++j) {
              if (!(x[j - 2] == a && x[j - 1] == b && x[j] == d)) continue;
              const int32_t f = x[j + 1];
              int32_t cnt = 0;
              int64_t last = -1;
              for (int64_t i = 2; i <= (int64_t)T - 2; ++i)
                if (x[i - 2] == a && x[i - 1] == b && x[i] == d && x[i + 1] == f) {
                  ++cnt;
                  last = i;
                }
              if (cnt > best_cnt || (cnt == best_cnt && last > best_last)) {
                found = 1;
                best_cnt = cnt;
                best_last = last;
                y = f;
              }
            }
            q = -1;
            run = 0;
            e = -best_cnt;
          }
        }
#undef CTX
        if (!found) break; /* nothing proposed */
        out[n] = y;
        ev[n] = e;
        ++n;
        ext[m++] = y;
      }
      ng_len[(int64_t)r * C + c] = n;
    }
  }
  free(ext);
  return status;
}

/* ------------------------------------------------------------------------ */
/* Budget sizing ([HS] sec. 2 adaptive verification, sec. 4.3 Eq. (2), sec. */
/* 4.4, App. F cost model, App. O stale sizing).  Over the slots that may   */
/* be verified (k < min(chain_len[r], max_verify_len)), with survivals     */
/* s_(1) >= s_(2) >= ... :                                                  */
/*   A(b) = batch + sum_{i <= b} s_(i)     (expected emitted tokens)        */
/*   C(b) = C0 + p b                       (App. F, the linear step cost)   */
/*   G(b) = A(b) / C(b);  b* = the smallest b in [0, #slots] maximising G;  */
/*   lambda = G(b*) p, the slot price of Eq. (2).                           */
/* The sums run in the sorted order, in double.  Reading: the eager-step    */
/* branch of App. F Eq. (4) is not modelled (one linear cost for every b).  */
/* ------------------------------------------------------------------------ */
static int cmp_desc_float(const void* a, const void* b) {
  const float x = *(const float*)a, y = *(const float*)b;
  return (x < y) - (x > y);
}

int oracle_size_budget(int32_t batch, int32_t L, const float* S, const int32_t* chain_len,
                       int32_t max_verify_len, double C0, double p, int32_t* b_star,
                       double* lambda, double* G_out) {
  if (batch < 0 || L < 1 || max_verify_len < 0 || !(C0 > 0.0) || !(p > 0.0)) return ORACLE_ERR_ARG;
  float* s = (float*)malloc(sizeof(float) * ((size_t)batch * L + 1));
  int32_t n = 0;
  for (int32_t r = 0; r < batch; ++r) {
    int32_t len = chain_len[r] < max_verify_len ? chain_len[r] : max_verify_len;
    if (len > L) len = L;
    for (int32_t k = 0; k < len; ++k) s[n++] = S[(int64_t)r * L + k];
  }
  qsort(s, (size_t)n, sizeof(float), cmp_desc_float);
  double A = (double)batch, best = A / C0;
  int32_t bs = 0;
  if (G_out) G_out[0] = best;
  for (int32_t b = 1; b <= n; ++b) {
    A += (double)s[b - 1];
    const double G = A / (C0 + p * (double)b);
    if (G_out) G_out[b] = G;
    if (G > best) {
      best = G;
      bs = b;
    }
  }
  *b_star = bs;
  *lambda = best * p;
  free(s);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Probabilistic drafting ([HS] sec. 4.5, App. H): the drafter's token at   */
/* position k (1-based) is drawn from q_k = softmax(z_k / T) over its       */
/* logit row, by inverse CDF in vocabulary order at the uniform u = word 0  */
/* of Philox4x32-10 with counter (r, 0x40000000 + k, lo32(step),            */
/* hi32(step)) and key (lo32(seed), hi32(seed)) -- a counter domain apart   */
/* from verification's (r, i <= 32, ...).  Reading: the positions are drawn */
/* independently from the given rows; a drafter whose logits depend on the  */
/* previous token (DSpark's Markov head) produces its rows inside its own   */
/* network.  A row holding NaN or +Inf is flagged and drafts its argmax.    */
/* ------------------------------------------------------------------------ */
int oracle_sample_drafts(int32_t batch, int32_t K, int32_t vocab, int32_t dtype,
                         const void* draft_logits, double temperature, uint64_t seed,
                         uint64_t step, const double* u_override, int32_t* y, double* dbg_u,
                         double* dbg_q) {
  if (batch < 0 || K < 1 || vocab < 1 || (dtype != 0 && dtype != 1) || !(temperature > 0.0))
    return ORACLE_ERR_ARG;
  int status = 0;
  double* q = (double*)malloc(sizeof(double) * (size_t)vocab);
  for (int32_t r = 0; r < batch; ++r)
    for (int32_t k = 1; k <= K; ++k) {
      const int64_t row = (int64_t)r * K + (k - 1);
      double u;
      if (u_override) {
        u = u_override[row];
      } else {
        uint32_t ctr[4] = {(uint32_t)r, 0x40000000u + (uint32_t)k, (uint32_t)step, (uint32_t)(step >> 32)};
        uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
        uint32_t out[4];
        oracle_philox4x32_10(ctr, key, out);
        u = oracle_u01(out[0]);
      }
      if (dbg_u) dbg_u[row] = u;
      if (row_nonfinite(draft_logits, row, vocab, dtype)) {
        status |= ORACLE_ST_NONFINITE;
        y[row] = row_argmax(draft_logits, row, vocab, dtype);
        if (dbg_q) dbg_q[row] = -1.0;
        continue;
      }
      row_softmax(draft_logits, row, vocab, dtype, temperature, q);
      const int32_t x = inverse_cdf(q, vocab, u);
      y[row] = x;
      if (dbg_q) dbg_q[row] = q[x];
    }
  free(q);
  return status;
}
