/*
 * spec.h -- C ABI of the GB300 (sm_103a) hot path of one hybrid
 * speculative-decoding round.
 *
 * One round runs four steps on one GPU, all on the caller's stream:
 *   1. spec_ngram_propose       n-gram prompt lookup over each request's history
 *   2. spec_price_and_allocate  Eq. (1) estimates, prefix survivals, chain choice
 *                               at slot price lambda, batch-wide budget allocation
 *   3. spec_verify_chain        verification of the chosen chains against the
 *                               target (and draft) distributions over the full
 *                               vocabulary, with Philox-driven rejection sampling
 *   4. spec_verify_tree         greedy verification of a candidate tree
 *
 * Sources (web pages, cited by title and section):
 *   [HS] "Hybrid Spark: Adaptive Speculative Decoding That Lets the Content
 *        Choose the Drafter" (arXiv 2611.05611v1)
 *   [AS] "AdaSpark: Adaptive DSpark with Online Learning for Tree Verification
 *        and N-gram Fill" (arXiv 2610.05774)
 *   [LS] "Efficient speculative decoding with a fixed-cost parallel drafter"
 *        (arXiv 2609.37029)
 *   [PH] Salmon et al., "Parallel random numbers: as easy as 1, 2, 3" (SC'11)
 *
 * Conventions for every entry point:
 *   - All array arguments are DEVICE pointers to caller-owned, contiguous,
 *     row-major buffers, except where a comment says "host".  The library
 *     allocates nothing and never synchronises with the host: every call only
 *     validates its scalar arguments on the host and enqueues kernels on
 *     `stream` ([HS] sec. 2 and 4.4: no host read of a GPU value mid-step).
 *   - The synchronous return value reports argument and launch errors only
 *     (SPEC_ERR_INVALID_ARG, SPEC_ERR_UNSUPPORTED, SPEC_ERR_WORKSPACE,
 *     SPEC_ERR_CUDA).  Data errors found on the device (an out-of-range token
 *     id, a NaN logit, a malformed tree, a length beyond a buffer) set bits in
 *     the workspace's 32-bit status word (SPEC_DEV_*), which the caller copies
 *     back asynchronously when it wants to; the affected request then gets a
 *     defined fallback output (documented per call) and the kernel returns
 *     normally.  Kernels never trap.
 *   - A workspace (caller-allocated device memory of spec_workspace_bytes()
 *     bytes, described by a host spec_workspace filled and zeroed once by
 *     spec_workspace_init()) carries the status word, per-request counters
 *     and per-row partial results.  Each call leaves its counters at zero
 *     again.  One workspace must not be used by two calls that may run
 *     concurrently (two streams).  Calls whose sizes exceed the workspace's
 *     capacity return SPEC_ERR_WORKSPACE.
 *   - Token ids are int32.  Lengths are int32.  Outputs beyond a request's
 *     valid length are filled with -1 (ids) or 0 (survivals, flags).
 */
#ifndef SPEC_H
#define SPEC_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SPEC_OK = 0,
  SPEC_ERR_INVALID_ARG = 1, /* a null pointer, a negative or inconsistent size  */
  SPEC_ERR_CUDA = 2,        /* a CUDA launch or runtime error                   */
  SPEC_ERR_UNSUPPORTED = 3, /* a size beyond the limits below                   */
  SPEC_ERR_WORKSPACE = 4    /* workspace missing, misaligned or too small       */
} spec_status;

typedef enum { SPEC_F32 = 0, SPEC_BF16 = 1 } spec_dtype;

/* chain-selection policies: [HS] sec. 4.3 (PROPOSED), sec. 4.5 and App. H
 * (NGRAM_FIRST, EXTENSION, lossless with probabilistic drafting), and the
 * two single-drafter baselines */
typedef enum {
  SPEC_POLICY_PROPOSED = 0,
  SPEC_POLICY_NGRAM_FIRST = 1,
  SPEC_POLICY_EXTENSION = 2,
  SPEC_POLICY_MODEL_ONLY = 3,
  SPEC_POLICY_NGRAM_ONLY = 4
} spec_policy;

/* source[] values written by spec_price_and_allocate */
#define SPEC_SRC_MODEL 0     /* the model drafter's chain d                      */
#define SPEC_SRC_NGRAM 1     /* the n-gram chain g                               */
#define SPEC_SRC_CONTAINS 2  /* g kept by the contains rule, survivals merged    */
#define SPEC_SRC_EXTENSION 3 /* d followed by g's tail (extension policy)        */

/* device status bits (OR-ed into the workspace status word) */
#define SPEC_DEV_BAD_TOKEN 0x1u  /* a draft token id outside [0, vocab): rejected    */
#define SPEC_DEV_NONFINITE 0x2u  /* NaN or +Inf in a logit row that was read         */
#define SPEC_DEV_BAD_TREE 0x4u   /* parent[0] != -1 or parent[j] outside [0, j)      */
#define SPEC_DEV_BAD_LENGTH 0x8u /* a length or row offset beyond its buffer         */
#define SPEC_DEV_BAD_VALUE 0x10u /* a confidence outside [0,1] (clamped), a feature
                                    outside the estimator table (h = 0)             */
#define SPEC_DEV_TIMEOUT 0x20u   /* a bounded wait on an asynchronous copy ran out  */
#define SPEC_DEV_OVERFLOW 0x40u  /* reserved: no call sets it (the n-gram fill
                                    counts any number of followers exactly)        */

/* limits */
#define SPEC_MAX_L 31            /* longest chain (L) and n-gram proposal           */
#define SPEC_MAX_N 32            /* largest n-gram match length n_max               */
#define SPEC_MAX_PRICE_BATCH 1024
#define SPEC_MAX_TREE_NODES 256
#define SPEC_MAX_TREE_CANDIDATES 512 /* the builder's 1 + P Kc + n_chains Lg      */
#define SPEC_MAX_COPY_CAP 4096
#define SPEC_MAX_VOCAB 524288    /* largest vocabulary of a workspace / logit row    */

const char* spec_status_string(spec_status s);
int32_t spec_version(void);

/* ------------------------------------------------------------------------
 * Workspace.
 * A spec_workspace is a small HOST struct (caller-owned) describing a
 * caller-allocated DEVICE buffer and the capacity it was laid out for:
 * at most `max_batch` requests, `max_rows` logit rows (row_off[batch] of a
 * chain layout or node_off[batch] of a tree batch), `K` model-drafter
 * positions and `vocab` entries per row.  The layout is fixed by
 * spec_workspace_init, so every call can use any sizes within the capacity.
 * spec_workspace_bytes: device bytes needed for that capacity (0 if invalid).
 * spec_workspace_init: fills *ws and zeroes the device buffer on `stream`
 *   (once, before first use).  dev_mem must be 256-byte aligned.
 * spec_workspace_status_word: device address of the 32-bit status word
 *   (the caller may copy it back, or reset it with cudaMemsetAsync).
 * ------------------------------------------------------------------------ */
typedef struct {
  void* base;            /* device buffer                                    */
  size_t bytes;          /* its size                                         */
  int32_t max_batch, max_rows, K, vocab;
  size_t off_counter;    /* uint32 [max_batch]: per-request arrival counters */
  size_t off_counter2;   /* uint32 [max_batch]: second-phase counters        */
  size_t off_record;     /* 64 B [max_batch]: resample records              */
  size_t off_rowkey;     /* uint64 [max_rows]: packed row argmax             */
  size_t off_partial;    /* float2 [(max_rows + max_batch K) x pstride]: per
                            chunk (max, sum) of a row, then the logit at its
                            draft token; pstride = units + 1 rounded up to
                            even                                             */
  size_t off_partial2;   /* float [max_batch x pstride]: per chunk residual
                            mass of a rejected position                    */
  size_t off_keys;       /* uint32 [SPEC_MAX_PRICE_BATCH x SPEC_MAX_L]:
                            allocation keys of the pricing step            */
  size_t off_counter3;   /* uint32 [max_batch x max(K, 1)]: per draft-row
                            arrival counters of spec_sample_drafts          */
  int32_t units;         /* ceil(vocab / 2048)                               */
  int32_t pad_;
} spec_workspace;

size_t spec_workspace_bytes(int32_t max_batch, int32_t max_rows, int32_t K, int32_t vocab);
spec_status spec_workspace_init(spec_workspace* ws, void* dev_mem, size_t bytes, int32_t max_batch,
                                int32_t max_rows, int32_t K, int32_t vocab, cudaStream_t stream);
uint32_t* spec_workspace_status_word(const spec_workspace* ws);

/* ------------------------------------------------------------------------
 * Eq. (1) estimator ([HS] sec. 4.2, App. D Table 5 coefficients):
 *   h_k = sigma(beta_k + w_pos(k) (n - n_ref) + delta a
 *               + [n = n_full] (ell_pos(k) + kappa_pos(k) ln(min(m, m_cap) / m_ref)))
 * with pos(k) = first for k = 1, rest otherwise.  Host struct.
 * ------------------------------------------------------------------------ */
typedef struct {
  double beta[32];               /* beta_k, k = 1..L, at beta[k-1]           */
  double w_first, w_rest;        /* match-length weights                      */
  double delta;                  /* agreement weight                          */
  double ell_first, ell_rest;    /* full-match bonus                          */
  double kappa_first, kappa_rest;/* copy-length weights                       */
  int32_t n_ref;                 /* 5                                         */
  int32_t n_full;                /* 15 (the n-gram drafter's n_max)           */
  int32_t m_cap;                 /* 256                                       */
  int32_t m_ref;                 /* 15                                        */
  int32_t use_constant_h;        /* 1: h_k = constant_h for every feature     */
  int32_t pad_;
  double constant_h;
} spec_estimator;

/* spec_estimator_table_bytes: bytes of the fp32 table of h over every
 *   (k, n, a, m) key for chains of up to L positions (0 on invalid input).
 * spec_estimator_build: evaluates Eq. (1) in double precision on the GPU for
 *   every key and stores each value rounded once to fp32 into `table`
 *   (device, 16-byte aligned, table_bytes >= spec_estimator_table_bytes).
 *   Done once per coefficient set; spec_price_and_allocate reads the table.
 *   `est` is host memory.  Keys: n in [0, SPEC_MAX_N], a in {0, 1},
 *   m in [0, m_cap] (m only enters when n = n_full). */
size_t spec_estimator_table_bytes(const spec_estimator* est, int32_t L);
spec_status spec_estimator_build(const spec_estimator* est, int32_t L, float* table,
                                 size_t table_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Step 1: n-gram prompt lookup ([HS] sec. 4.1, sec. 4.2 feature list,
 * sec. 5.1: the longest match is the one used).
 *
 * For request r with history x = hist[r * hist_stride ...], T = hist_len[r]:
 * every earlier end position j <= T-2 has a match length l(j), the length of
 * the common suffix of x[..j] and x[..T-1], capped at copy_cap (and at j+1).
 * Candidates have l(j) >= n_min and are ranked by (l(j), j) descending (the
 * longest copy wins; equal lengths go to the most recent occurrence).  For
 * the best j*:
 *   g[r, 0..g_len)  = x[j*+1 .. j*+g_len], g_len = min(max_propose, T-1-j*)
 *   match_n[r]      = min(l(j*), n_max)                        (n)
 *   agree[r]        = 1 if there is no runner-up or the runner-up's next
 *                     token equals x[j*+1], else 0             (a)
 *   copy_len[r]     = l(j*)                                    (m)
 * No candidate: g_len = n = a = m = 0.  g is [batch x max_propose], unused
 * entries -1.  hist_len[r] outside [0, hist_stride] sets SPEC_DEV_BAD_LENGTH
 * and gives the no-candidate output.
 * Limits: 1 <= n_min <= n_max <= SPEC_MAX_N, n_max <= copy_cap <=
 * SPEC_MAX_COPY_CAP, 0 <= max_propose <= SPEC_MAX_L, hist_stride <= 393216.
 * ------------------------------------------------------------------------ */
spec_status spec_ngram_propose(const int32_t* hist, int64_t hist_stride, const int32_t* hist_len,
                               int32_t batch, int32_t n_min, int32_t n_max, int32_t max_propose,
                               int32_t copy_cap, int32_t* g, int32_t* g_len, int32_t* match_n,
                               int32_t* agree, int32_t* copy_len, const spec_workspace* ws,
                               cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Step 2: pricing, chain choice and batch-wide allocation ([HS] Algorithm 1;
 * sec. 4.2; sec. 4.3 Eq. (2)-(3), contains rule; sec. 4.4; sec. 4.5 and
 * App. H policies; sec. 2 adaptive verification).
 *
 * Per request r (d: [batch x K] model chain with d_len[r] <= K tokens and
 * confidences c [batch x K] in [0,1]; g, g_len, match_n, agree, copy_len:
 * the outputs of step 1 with g [batch x L]):
 *   h_k  = table value of Eq. (1) for (k, n, a, m)          (fp32)
 *   S^g_k = S^g_{k-1} * h_k,  S^d_k = S^d_{k-1} * c_k        (fp32, k order)
 *   V    = sum_k max(S_k - lambda, 0)                        (fp32, k order)
 *   PROPOSED: contains rule if d_len >= 1, g_len > d_len and g starts with
 *     all of d: chain g, S_k = max(S^g_k, S^d_k) for k <= d_len, then
 *     S_k = S_{k-1} * h_k; else g if g_len > 0 and V^g >= V^d; else d.
 *   NGRAM_FIRST: g if g_len > 0 else d.  EXTENSION: d, followed by g's tail
 *     when d (d_len >= 1) is a proper prefix of g; tail survivals continue
 *     from S^d and tail slots are point masses.  MODEL_ONLY: d.  NGRAM_ONLY: g.
 *   point_mass[r, k] = 1 for n-gram tokens, and for model tokens when
 *     draft_greedy != 0 (greedy drafting); 0 for sampled model tokens.
 * Allocation: among the slots (r, k), k < min(chain_len[r], max_verify_len),
 * the min(budget, #slots) slots with the highest S (ties: lower r, then
 * lower k) are verified; each request keeps a prefix of length verify_len[r].
 * row_off[0] = 0, row_off[r+1] = row_off[r] + verify_len[r] + 1 (the verify
 * layout: request r's target rows are row_off[r] .. row_off[r] + verify_len[r]).
 * lambda and budget are host scalars ([HS] sec. 4.4).
 * Outputs: chain [batch x L] (-1 past chain_len), S [batch x L] (0 past),
 * chain_len, source (SPEC_SRC_*), verify_len [batch], row_off [batch + 1],
 * point_mass uint8 [batch x L].
 * est_table: built by spec_estimator_build from `est` (host) for this L;
 * est_table_bytes < spec_estimator_table_bytes(est, L) is SPEC_ERR_INVALID_ARG.
 * Limits: 1 <= L <= SPEC_MAX_L, 0 <= K <= L, batch <= SPEC_MAX_PRICE_BATCH.
 * ------------------------------------------------------------------------ */
spec_status spec_price_and_allocate(
    int32_t batch, int32_t K, int32_t L, const int32_t* d, const float* c, const int32_t* d_len,
    const int32_t* g, const int32_t* g_len, const int32_t* match_n, const int32_t* agree,
    const int32_t* copy_len, const spec_estimator* est, const float* est_table,
    size_t est_table_bytes, float lambda,
    int32_t budget, int32_t max_verify_len, spec_policy policy, int32_t draft_greedy,
    int32_t* chain, float* S, int32_t* chain_len, int32_t* source, int32_t* verify_len,
    int32_t* row_off, uint8_t* point_mass, const spec_workspace* ws, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Steps 1 + 2 fused: spec_ngram_propose followed by spec_price_and_allocate
 * in one launch, with identical outputs (every argument has the meaning it has
 * in those two calls; max_propose = L).  Each request's n-gram CTA prices its
 * own request from on-chip values (the n-gram scan already yields the Eq. (1)
 * features n, a and m, [HS] sec. 4.2), and the last request to finish
 * allocates the budget for the batch.  Limits: those of both calls.
 * ------------------------------------------------------------------------ */
spec_status spec_draft_and_price(
    const int32_t* hist, int64_t hist_stride, const int32_t* hist_len, int32_t batch, int32_t n_min,
    int32_t n_max, int32_t copy_cap, int32_t* g, int32_t* g_len, int32_t* match_n, int32_t* agree,
    int32_t* copy_len, int32_t K, int32_t L, const int32_t* d, const float* c, const int32_t* d_len,
    const spec_estimator* est, const float* est_table, size_t est_table_bytes, float lambda,
    int32_t budget, int32_t max_verify_len, spec_policy policy, int32_t draft_greedy, int32_t* chain,
    float* S, int32_t* chain_len, int32_t* source, int32_t* verify_len, int32_t* row_off,
    uint8_t* point_mass, const spec_workspace* ws, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * spec_ngram_fill: the n-gram chains of a candidate tree ([AS] sec. 2.2, the
 * chains that branch from the anchor and from each pick and may run past the
 * drafter's block; sec. 3.3 "N-gram candidates"; the parameter table's
 * three-token follower context and 32-token depth).  Its output is
 * spec_build_tree's chain input with n_chains = P + 1.
 *
 * Per request r the committed text x = hist[r][0 .. hist_len[r]-1] (row
 * stride hist_stride) ends with the anchor.  Chain 0 starts at the anchor
 * and chain c >= 1 at pick c-1 = cand_tok[r][c-1][0] (cand_tok
 * [batch x P x Kc], the builder's block), with context ctx = x followed by
 * pick_0 .. pick_{c-1}.  Each step appends one token y to the chain and ctx:
 *   1. while reading along an earlier passage whose next position is
 *      <= T-1, y is that token;
 *   2. else, over end positions j <= T-2 with l(j) = common-suffix length of
 *      x[..j] and ctx (capped at copy_cap and j+1) >= n_min, the largest
 *      (l, j): y = x[j+1], and the chain reads on along x from j+2;
 *   3. else the most frequent follower x[j+1] of ctx's last three tokens over
 *      j in [2, T-2] (ties: the follower seen most recently);
 *   4. else the chain stops.
 * A chain stops at depth max_depth below the anchor (pick c-1 sits at depth
 * c), so chain c holds at most min(Lg, max_depth - c) tokens.
 * Outputs: ng_tok [batch x (P+1) x Lg] (-1 past each chain), ng_len
 * [batch x (P+1)], ng_ev [batch x (P+1) x Lg] (each token's evidence: the
 * length of the copy it continues, capped at copy_cap, for steps 1-2; minus
 * the follower's count for step 3; 0 past the chain).
 * hist_len[r] outside [0, hist_stride] sets SPEC_DEV_BAD_LENGTH (no chains).
 * Any number of distinct followers is counted exactly (a context with more
 * than 2048 takes extra passes over the text).  Limits: P >= 0, Kc >= 1, 1 <= n_min <= copy_cap,
 * max_depth >= 0, Lg >= 0, P + Lg <= 4096, batch <= 65535.  The workspace
 * serves only its status word.
 * ------------------------------------------------------------------------ */
spec_status spec_ngram_fill(const int32_t* hist, int64_t hist_stride, const int32_t* hist_len, int32_t batch,
                            int32_t P, int32_t Kc, const int32_t* cand_tok, int32_t n_min, int32_t copy_cap,
                            int32_t max_depth, int32_t Lg, int32_t* ng_tok, int32_t* ng_len, int32_t* ng_ev,
                            const spec_workspace* ws, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * spec_build_tree: the candidate tree of one block-drafter round ([AS]
 * sec. 2.2 tree shape; sec. 3.3 n-gram candidates and Eq. (6); sec. 3.1 and
 * Proposition 1, best-first order; Algorithm 1, the first n-1 nodes laid out
 * depth-first).  Its output feeds spec_verify_tree.
 *
 * Per request r: anchor[r], the committed token the tree hangs from; a block
 * of P positions with Kc ranked candidates each, cand_tok / cand_score
 * [batch x P x Kc] (k = 0 the drafter's pick, k >= 1 its siblings; the score
 * s of Eq. (6), from the caller's acceptance model); n_chains n-gram chains,
 * ng_tok [batch x n_chains x Lg] with ng_len[r][c] tokens, chain 0 from the
 * anchor and chain c >= 1 from pick c-1 (1 <= n_chains <= P + 1; the layout
 * spec_ngram_fill writes); ng_score[r], the score of an n-gram node;
 * ng_adj[r] = max(0, logit p_src), added to an agreed drafter candidate's
 * score and subtracted from a contradicted one's.
 * Candidates: 0 the anchor; 1 + i Kc + k position i's k-th candidate; then
 * the n-gram nodes in the order the chains make them.  Pick i hangs from
 * pick i-1 (pick 0 from the anchor); the siblings of position i hang from
 * the pick's parent, as leaves.  The chains walk in order c = 0, 1, ...: a
 * step equal to a drafter child of the current node marks that child agreed
 * (lowest index on duplicates) and moves to it; else a step equal to an
 * n-gram child already there moves to it; else it appends an n-gram node and
 * moves to it.  The other drafter children of every node a chain passes
 * through are contradicted, unless some chain agrees with them.
 * Scores are clamped to [-80, 80].
 * q_j = e^{s_j} / (1 + sum over the children c of parent(j) of e^{s_c}),
 * Q_j = Q_parent(j) q_j (fp64); order: Q descending, ties to the lower index.
 * Outputs [batch x width]: the anchor and the first width-1 candidates of the
 * order, depth-first with children in increasing candidate index: tok,
 * parent (row of the parent, -1 at the anchor), cand_id (candidate index);
 * rows past n_rows[r] = min(width, number of candidates) are -1.
 * ng_len[r][c] outside [0, Lg] sets SPEC_DEV_BAD_LENGTH (that chain is empty).
 * Limits: Kc >= 1, P >= 0, Lg >= 0, 1 + P Kc + n_chains Lg <=
 * SPEC_MAX_TREE_CANDIDATES, 1 <= width <= SPEC_MAX_TREE_NODES.  The workspace
 * serves only its status word.
 * ------------------------------------------------------------------------ */
spec_status spec_build_tree(int32_t batch, int32_t P, int32_t Kc, const int32_t* anchor,
                            const int32_t* cand_tok, const float* cand_score, const int32_t* ng_tok,
                            int32_t n_chains, int32_t Lg, const int32_t* ng_len, const float* ng_score,
                            const float* ng_adj, int32_t width, int32_t* tok, int32_t* parent, int32_t* cand_id,
                            int32_t* n_rows, const spec_workspace* ws, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * spec_sample_drafts: probabilistic drafting ([HS] sec. 4.5 and App. H;
 * the drafter samples its tokens from its own distribution q).
 *
 * draft_logits [batch x K x vocab] (fp32 or bf16) holds the drafter's logit
 * row of every position; y [batch x K] gets y[r, k-1] ~ q_k = softmax(z / T)
 * by inverse CDF in vocabulary order at the uniform u = word 0 of
 * Philox4x32-10 with counter (r, 0x40000000 + k, lo32(step), hi32(step)) and
 * key (lo32(seed), hi32(seed)) -- a counter domain apart from
 * spec_verify_chain's.  The positions are drawn independently from the given
 * rows (a drafter whose row depends on the previous token produces its rows
 * inside its own network).  dbg_u / dbg_q [batch x K] (may be NULL): the
 * uniform and q of the drawn token.  The rows' per-chunk (max, sum) are left
 * in workspace slots apart from the target rows'.
 * T must be > 0.  A row holding NaN or +Inf sets SPEC_DEV_NONFINITE.
 * Limits: batch <= the workspace's max_batch and <= 2048, 1 <= K <= its K,
 * vocab <= its vocab.
 * ------------------------------------------------------------------------ */
spec_status spec_sample_drafts(int32_t batch, int32_t K, int32_t vocab, spec_dtype dtype,
                               const void* draft_logits, float temperature, uint64_t seed, uint64_t step,
                               int32_t* y, float* dbg_u, float* dbg_q, const spec_workspace* ws,
                               cudaStream_t stream);

/* ------------------------------------------------------------------------
 * spec_size_budget: the next verification budget and slot price from one
 * step's survivals ([HS] sec. 2 adaptive verification, sec. 4.3 Eq. (2),
 * sec. 4.4, App. F cost model, App. O stale sizing).
 *
 * Over the slots (r, k) with k < min(chain_len[r], max_verify_len), whose
 * survivals S [batch x L] are the output of spec_price_and_allocate, sorted
 * descending s_(1) >= s_(2) >= ...:
 *   G(b) = (batch + sum_{i <= b} s_(i)) / (C0 + p b)   (fp64),
 *   *out_budget = b*, the smallest maximiser of G over b in [0, #slots],
 *   *out_lambda = G(b*) p, rounded to fp32.
 * C0 (base step cost) and p (cost of one verification slot) are host
 * scalars from the caller's cost model (App. F); only their ratio matters.
 * The host reads the two device scalars back asynchronously and passes them
 * as `budget` and `lambda` to the pricing step two steps later ([HS] sec.
 * 4.4: the GPU allocates from fresh survivals, the host sizes from stale
 * ones).  The maximum is found without sorting, by Dinkelbach's iteration on
 * the ratio (the set that maximises A - lambda C takes every slot above
 * lambda p), with the survivals summed exactly in 2^-48 fixed point, so
 * near-ties of G may resolve differently from a left-to-right fp64 sum in
 * the last bits.  A survival outside [0, 1] (or NaN) among the verifiable
 * slots sets SPEC_DEV_BAD_VALUE and counts as clamped to [0, 1] (NaN as 0).
 * The workspace serves only its status word (the call may overlap other
 * calls on it).
 * Limits: 1 <= L <= SPEC_MAX_L, batch <= SPEC_MAX_PRICE_BATCH; C0, p > 0.
 * ------------------------------------------------------------------------ */
spec_status spec_size_budget(int32_t batch, int32_t L, const float* S, const int32_t* chain_len,
                             int32_t max_verify_len, double C0, double p, int32_t* out_budget,
                             float* out_lambda, const spec_workspace* ws, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * spec_price_and_allocate_static: step 2 without a workspace.  The method has
 * no counterpart of this call; it is an interface variant of
 * spec_price_and_allocate for callers that cannot hand the library device
 * memory -- for example a scheduler whose device memory is planned up front
 * and that may not allocate while a decoding step is in flight, or a host
 * thread that must not call into an allocator.  Every argument except
 * `status_word` has its meaning in spec_price_and_allocate, and the outputs
 * are identical to that call's on the same inputs.
 *
 * Scratch: a fixed array of (64 + SPEC_STATIC_PRICE_MAX_BATCH * SPEC_MAX_L)
 * 32-bit words (32,000 bytes) in this library's device memory; this call and
 * its kernel allocate nothing.
 * Set-up: the first call in each context looks up that array's device
 * address (cudaGetSymbolAddress, with the device current) and keeps it with
 * the context's process-unique id (cuCtxGetId); a call from another context
 * -- after cudaDeviceReset, or from a driver-API context on the same device --
 * looks it up again, so no kept address outlives its context.  Make the first
 * call in a context before the stream is captured into a graph.
 * Limits: batch <= SPEC_STATIC_PRICE_MAX_BATCH, else SPEC_ERR_UNSUPPORTED
 * before any device work; the other limits of spec_price_and_allocate.
 * Zero state: the array's arrival counter must be zero when a call's kernel
 * starts; it is zero when the library's device code loads into a context, and
 * every call whose kernel runs to completion leaves it at zero.  A kernel cut
 * off part way (a sticky CUDA error) leaves the context unusable; the context
 * that replaces it starts from a zeroed array.  The allocation keys need no
 * initial value.
 * Concurrency: every call on one device shares the one array, so calls whose
 * kernels may overlap on the device (different streams without an order
 * between them, or several host threads) race; keep them in one stream order.
 * status_word: device address of a caller-owned 32-bit word into which device
 * errors are OR-ed (SPEC_DEV_*), or NULL to discard them.
 * ------------------------------------------------------------------------ */
#define SPEC_STATIC_PRICE_MAX_BATCH 256
spec_status spec_price_and_allocate_static(
    int32_t batch, int32_t K, int32_t L, const int32_t* d, const float* c, const int32_t* d_len,
    const int32_t* g, const int32_t* g_len, const int32_t* match_n, const int32_t* agree,
    const int32_t* copy_len, const spec_estimator* est, const float* est_table,
    size_t est_table_bytes, float lambda,
    int32_t budget, int32_t max_verify_len, spec_policy policy, int32_t draft_greedy,
    int32_t* chain, float* S, int32_t* chain_len, int32_t* source, int32_t* verify_len,
    int32_t* row_off, uint8_t* point_mass, uint32_t* status_word, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Step 3: chain verification ([HS] sec. 2: the target keeps the longest
 * draft prefix that survives rejection sampling and adds one token of its
 * own; App. H point masses;
 * [LS] sec. 2.1: accept y_i with probability min(1, p_i(y_i)/q_i(y_i)), at the
 * first rejection draw from norm(max(0, p_i - q_i)), after B acceptances draw
 * a bonus from p_{B+1}; r accepted => r + 1 tokens).
 *
 * Request r verifies ell = verify_len[r] drafts y = chain[r, 0..ell).  Its
 * target logit rows are target_logits[row_off[r] + i], i = 0..ell (row i
 * holds position i+1; row ell the bonus position); they must satisfy
 * row_off[r] + ell < row_off[r+1] <= row_off[batch] <= max_rows, so both the
 * compact layout of step 2 and a strided layout (row_off[r] = r * rows) work.
 * target_logits holds row_off[batch] rows of `vocab` entries (fp32 or bf16).
 * T = temperature:
 *   T <= 0: greedy target.  Accept y_i iff y_i = argmax z_i (lowest index on
 *     ties); the first failure emits argmax z_i; all accepted emit argmax z_ell.
 *   T > 0: p_i = softmax(z_i / T).  q_i = softmax(draft_logits[r, i-1] / T)
 *     when point_mass[r, i-1] == 0 (requires i <= K and draft_logits), else
 *     q_i = delta_{y_i}.  u_i, u'_i = words 0 and 1 of Philox4x32-10 [PH]
 *     with key (lo32(seed), hi32(seed)) and counter (r, i, lo32(step),
 *     hi32(step)), each mapped to (w >> 8) * 2^-24.  Accept iff
 *     ratio = p_i(y_i)/q_i(y_i) >= 1 or u_i < ratio.  At the first rejection
 *     the emitted token is the smallest x (vocabulary order) whose running
 *     sum of r = max(0, p_i - q_i) (p_i with y_i removed for a point mass)
 *     exceeds u'_i * sum(r); a residual of total mass <= 1e-30 is replaced by
 *     p_i.  All accepted: the bonus is drawn from p_{ell+1} with u'_{ell+1}.
 * Outputs: out_tokens [batch x (L+1)] (the n_accepted drafts, then the
 * correction or bonus token, then -1), n_accepted, n_emitted = n_accepted + 1.
 * Optional (NULL to skip): dbg_ratio, dbg_u [batch x L] (-1 where untested),
 * dbg_resid [batch] (probability of the emitted correction / bonus under its
 * normalised residual; 1 at T <= 0).
 * Invalid request (layout, verify_len > L): SPEC_DEV_BAD_LENGTH,
 * n_accepted = n_emitted = 0 and no tokens.  A draft id outside [0, vocab)
 * sets SPEC_DEV_BAD_TOKEN and is rejected.
 * Limits: L <= SPEC_MAX_L, 1 <= vocab <= SPEC_MAX_VOCAB, batch <= 2048,
 * (max_rows + batch K) x ceil(vocab / chunk) < 2^31 with chunk = 4096 (bf16)
 * or 2048 (fp32) entries; else SPEC_ERR_UNSUPPORTED.
 * Launches: one kernel streams every row once and finalises each request;
 * with draft distributions (T > 0), a second kernel makes the draws from
 * max(0, p_i - q_i) of the requests that reject a drafted token (it reads
 * the two rows again, from L2).
 * ------------------------------------------------------------------------ */
spec_status spec_verify_chain(
    int32_t batch, int32_t vocab, spec_dtype dtype, const void* target_logits,
    const int32_t* row_off, int32_t max_rows, const void* draft_logits, int32_t K,
    const int32_t* chain, int32_t L, const int32_t* verify_len, const uint8_t* point_mass,
    float temperature, uint64_t seed, uint64_t step, int32_t* out_tokens, int32_t* n_accepted,
    int32_t* n_emitted, float* dbg_ratio, float* dbg_u, float* dbg_resid,
    const spec_workspace* ws, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * spec_verify_chain_drafted: spec_verify_chain, with the same arguments and
 * the same results, when the draft distributions come from
 * spec_sample_drafts on the same workspace.  That call left each draft row's
 * per-chunk (max, sum) statistics and the logit at its drawn token in the
 * workspace; this one uses them instead of reading the draft rows again, so
 * it streams only the target rows (the draft rows are still read, from L2,
 * by the max(0, p - q) draw at a rejection).
 * Requires: draft_logits, K, vocab, dtype and temperature equal to that
 * spec_sample_drafts call's; for every position with point_mass == 0, the
 * chain holds the token that call drew (as spec_draft_and_price places it);
 * no call that writes draft-row statistics (spec_sample_drafts or
 * spec_verify_chain with draft_logits) on the same workspace in between.
 * draft_logits, point_mass and temperature > 0 are required
 * (SPEC_ERR_INVALID_ARG).  A temperature other than the drafting call's sets
 * SPEC_DEV_BAD_VALUE.
 * ------------------------------------------------------------------------ */
spec_status spec_verify_chain_drafted(
    int32_t batch, int32_t vocab, spec_dtype dtype, const void* target_logits,
    const int32_t* row_off, int32_t max_rows, const void* draft_logits, int32_t K,
    const int32_t* chain, int32_t L, const int32_t* verify_len, const uint8_t* point_mass,
    float temperature, uint64_t seed, uint64_t step, int32_t* out_tokens, int32_t* n_accepted,
    int32_t* n_emitted, float* dbg_ratio, float* dbg_u, float* dbg_resid,
    const spec_workspace* ws, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Step 4: greedy tree verification ([AS] sec. 2.2, sec. 3.5).
 *
 * Request r's tree has n = node_off[r+1] - node_off[r] nodes (1 <= n <=
 * max_nodes) at rows node_off[r] + j of `logits`; node 0 is the anchor
 * (parent -1), parent[node_off[r] + j] in [0, j) is local, tok[...] is the
 * node's token.  a_j = argmax of row j (lowest index on ties).  Walking from
 * the anchor, the next node is the lowest-index child whose token equals the
 * current node's argmax; the walk stops when no child matches.
 * Outputs: path [batch x max_nodes] (local node indices, anchor first, then
 * -1), accept_len[r] = |path| - 1, out_tokens [batch x max_nodes] (tokens of
 * the accepted nodes, then the argmax at the last one, then -1).
 * A malformed tree sets SPEC_DEV_BAD_TREE (n outside [1, max_nodes]:
 * SPEC_DEV_BAD_LENGTH) and gives accept_len = -1 with no tokens.
 * Limits: max_nodes <= SPEC_MAX_TREE_NODES, node_off[batch] <= max_rows,
 * 1 <= vocab <= SPEC_MAX_VOCAB, batch <= 2048.
 * ------------------------------------------------------------------------ */
spec_status spec_verify_tree(int32_t batch, int32_t vocab, spec_dtype dtype, const void* logits,
                             const int32_t* node_off, int32_t max_rows, const int32_t* tok,
                             const int32_t* parent, int32_t max_nodes, int32_t* path,
                             int32_t* accept_len, int32_t* out_tokens,
                             const spec_workspace* ws, cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* SPEC_H */
