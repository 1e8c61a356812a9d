// tree.cu -- the candidate tree of one block-drafter round.
//
// AdaSpark sec. 2.2 (tree shape), sec. 3.3 (n-gram candidates, Eq. (6)),
// sec. 3.1 with Proposition 1 (best-first order) and Algorithm 1 (the first
// n-1 nodes of the order, laid out depth-first):
//   candidates: 0 the anchor; 1 + i Kc + k the k-th ranked candidate of block
//     position i (k = 0 the pick); pick i hangs from pick i-1 (pick 0 from the
//     anchor), the siblings of position i from the pick's parent, as leaves;
//   the n-gram chain walks from the anchor: a step equal to a drafter child of
//     the current node marks it agreed (lowest index on duplicates) and moves
//     to it, else it appends an n-gram node; the other drafter children of
//     every node it passes through are contradicted;
//   s: the given drafter score + adj if agreed - adj if contradicted, or the
//     n-gram score; clamped to [-80, 80];
//   q_j = e^{s_j} / (1 + sum over the children c of parent(j) of e^{s_c})
//     (children summed in index order), Q_j = Q_parent(j) q_j, in fp64;
//   order: Q descending, ties to the lower index; the tree: the anchor and the
//     first width-1 candidates, depth-first with children in index order.
//
// GB300 layout: one CTA per request, one thread per candidate (at most 256),
// everything in shared memory.  Warp 0 merges the n-gram chain (sequential in
// its steps, lane-parallel over a node's children).  A node's children are a
// known index range of drafter candidates plus at most one n-gram node, so the
// per-parent sums and the depth-first offsets cost O(Kc) per node; the rank of
// every candidate is a count over all candidates, the subtree sizes come from
// shared-memory atomics along each path, and Q is formed level by level from
// the anchor, one barrier per tree level.
#include "common.cuh"

namespace spec {

#define TB_THREADS 256

struct TreeParams {
  int32_t batch, P, Kc, Lg, width;
  const int32_t* anchor;
  const int32_t* cand_tok;
  const float* cand_score;
  const int32_t* ng_tok;
  const int32_t* ng_len;
  const float* ng_score;
  const float* ng_adj;
  int32_t* tok;
  int32_t* parent;
  int32_t* cand_id;
  int32_t* n_rows;
  uint32_t* status;
};

__global__ void __launch_bounds__(TB_THREADS) build_tree_kernel(TreeParams p) {
  __shared__ int32_t s_tok[TB_THREADS], s_par[TB_THREADS], s_flag[TB_THREADS];
  __shared__ double s_e[TB_THREADS], s_den[TB_THREADS], s_Q[TB_THREADS];
  __shared__ int32_t s_sel[TB_THREADS], s_size[TB_THREADS], s_before[TB_THREADS];
  __shared__ int32_t s_chain[TB_THREADS];
  __shared__ int32_t s_N, s_maxd, s_ngc, s_gl;
  __shared__ float s_ngs, s_adj;
  const int r = blockIdx.x, j = threadIdx.x;
  const int P = p.P, Kc = p.Kc;
  const int ND = 1 + P * Kc;  // anchor + drafter candidates
  // every global input of the request, loaded at once: the drafter's block,
  // its scores, the chain and the per-request scalars
  float my_score = 0.0f;
  if (j < ND) {
    if (j == 0) {
      s_tok[0] = p.anchor[r];
      s_par[0] = -1;
      s_gl = p.ng_len[r];
      s_ngs = p.ng_score[r];
      s_adj = p.ng_adj[r];
    } else {
      const int i = (j - 1) / Kc;
      s_tok[j] = p.cand_tok[(int64_t)r * P * Kc + (j - 1)];
      my_score = p.cand_score[(int64_t)r * P * Kc + (j - 1)];
      s_par[j] = (i == 0) ? 0 : 1 + (i - 1) * Kc;
    }
    s_flag[j] = 0;
  }
  s_size[j] = 0;
  if (j == 0) s_maxd = 0;
  // the chain's tokens, staged for the sequential walk below
  if (j < p.Lg) s_chain[j] = p.ng_tok[(int64_t)r * p.Lg + j];
  __syncthreads();
  // the n-gram chain from the anchor, by warp 0: each step depends on where
  // the previous one went (lanes compare the current node's drafter children
  // at once); once the chain leaves the drafter's block it only appends
  // n-gram nodes, which the warp writes in parallel
  if (j < 32) {
    const int lane = j;
    int32_t gl = s_gl;
    if (gl < 0 || gl > p.Lg) {
      if (lane == 0) set_status(p.status, SPEC_DEV_BAD_LENGTH);
      gl = 0;
    }
    int32_t cur = 0;                  // current node
    int32_t c0 = (P > 0) ? 1 : -1;    // its drafter children [c0, c0 + Kc), -1: none
    int32_t pos = 0;                  // the block position of those children
    int32_t t = 0;
    for (; t < gl && c0 >= 0; ++t) {
      const int32_t x = s_chain[t];
      // the lowest-index drafter child with token x
      int32_t hit = -1;
      for (int32_t k0 = 0; k0 < Kc && hit < 0; k0 += 32) {
        const int32_t k = k0 + lane;
        const unsigned b = __ballot_sync(0xFFFFFFFFu, k < Kc && s_tok[c0 + k] == x);
        if (b != 0u) hit = c0 + k0 + __ffs(b) - 1;
      }
      for (int32_t k = lane; k < Kc; k += 32)
        if (c0 + k != hit) s_flag[c0 + k] = -1;
      if (hit < 0) break;  // appended below, with every later step
      if (lane == 0) s_flag[hit] = 1;
      cur = hit;
      // a pick's children are the next position's candidates; a sibling has none
      const bool pick = (hit - c0) == 0;
      ++pos;
      c0 = (pick && pos < P) ? 1 + pos * Kc : -1;
    }
    // steps t .. gl-1 append a chain of n-gram nodes under cur
    const int32_t rest = gl - t;
    for (int32_t k = lane; k < rest; k += 32) {
      s_tok[ND + k] = s_chain[t + k];
      s_par[ND + k] = (k == 0) ? cur : ND + k - 1;
      s_flag[ND + k] = 0;
    }
    if (lane == 0) {
      s_N = ND + rest;
      s_ngc = rest > 0 ? cur : -1;  // the node the n-gram nodes hang from
    }
  }
  __syncthreads();
  const int N = s_N;
  // scores and e^s
  if (j >= 1 && j < N) {
    double s;
    if (j < ND) {
      const double adj = (double)s_adj;
      s = (double)my_score;
      s += (s_flag[j] > 0 ? adj : 0.0) - (s_flag[j] < 0 ? adj : 0.0);
    } else {
      s = (double)s_ngs;
    }
    s = s > 80.0 ? 80.0 : (s < -80.0 ? -80.0 : s);
    s_e[j] = exp(s);
  }
  __syncthreads();
  // every node's children: a range of Kc drafter candidates (under the anchor
  // and under a pick that is not the last) and at most one n-gram node (the
  // chain passes each node once); both in increasing index
  const int32_t ngc = s_ngc;
  auto drafter_kids = [&](int32_t v) -> int32_t {  // first drafter child, or -1
    if (v == 0) return P > 0 ? 1 : -1;
    if (v < ND && (v - 1) % Kc == 0 && (v - 1) / Kc + 1 < P) return v + Kc;
    return -1;
  };
  auto ngram_kid = [&](int32_t v) -> int32_t {  // the n-gram child, or -1
    if (v == ngc) return ND;
    return (v >= ND && v + 1 < N) ? v + 1 : -1;
  };
  // Eq. (6) denominators: thread j sums its own children in index order
  if (j < N) {
    double den = 1.0;
    const int32_t c0 = drafter_kids(j);
    if (c0 >= 0)
      for (int32_t k = 0; k < Kc; ++k) den += s_e[c0 + k];
    const int32_t g = ngram_kid(j);
    if (g >= 0) den += s_e[g];
    s_den[j] = den;
  }
  __syncthreads();
  // q_j, depths, then Q_j = Q_parent(j) q_j level by level from the anchor
  // down (the order of the definition's products)
  double qj = 1.0;
  int32_t dj = 0;
  if (j < N) {
    if (j > 0) qj = s_e[j] / s_den[s_par[j]];
    for (int32_t a = j; a != 0; a = s_par[a]) ++dj;
    atomicMax(&s_maxd, dj);
  }
  if (j == 0) s_Q[0] = 1.0;
  __syncthreads();
  const int32_t maxd = s_maxd;
  for (int32_t d = 1; d <= maxd; ++d) {
    if (j < N && dj == d) s_Q[j] = s_Q[s_par[j]] * qj;
    __syncthreads();
  }
  // best-first rank (Q descending, ties to the lower index) and selection
  if (j < N) {
    bool sel = (j == 0);
    if (j > 0) {
      // Q >= 0, so its bit pattern orders like its value: integer compares
      // (fp64 compares run on the narrow FP64 pipe)
      const unsigned long long kj = (unsigned long long)__double_as_longlong(s_Q[j]);
      int32_t rank = 0;
#pragma unroll 8
      for (int32_t i = 1; i < N; ++i) {
        const unsigned long long ki = (unsigned long long)__double_as_longlong(s_Q[i]);
        rank += (ki > kj || (ki == kj && i < j)) ? 1 : 0;
      }
      sel = rank < p.width - 1;
    }
    s_sel[j] = sel ? 1 : 0;
    // the selected subtree sizes: every selected node counts itself and its
    // ancestors (a prefix of the order is a tree, so they are selected too)
    if (sel)
      for (int32_t a = j;; a = s_par[a]) {
        atomicAdd(&s_size[a], 1);
        if (a == 0) break;
      }
  }
  __syncthreads();
  // before[c]: the rows that the selected earlier siblings of c occupy
  if (j < N && s_sel[j]) {
    int32_t run = 0;
    const int32_t c0 = drafter_kids(j);
    if (c0 >= 0)
      for (int32_t k = 0; k < Kc; ++k)
        if (s_sel[c0 + k]) {
          s_before[c0 + k] = run;
          run += s_size[c0 + k];
        }
    const int32_t g = ngram_kid(j);
    if (g >= 0 && s_sel[g]) s_before[g] = run;
  }
  __syncthreads();
  // depth-first position: one row per ancestor step, plus the earlier
  // siblings' subtrees at every level
  const int32_t n_rows = s_size[0];
  if (j < N && s_sel[j]) {
    int32_t pos = 0;
    for (int32_t a = j; a != 0; a = s_par[a]) pos += 1 + s_before[a];
    const int64_t o = (int64_t)r * p.width + pos;
    p.tok[o] = s_tok[j];
    p.parent[o] = (j == 0) ? -1 : pos - 1 - s_before[j];
    p.cand_id[o] = j;
  }
  for (int32_t z = n_rows + j; z < p.width; z += TB_THREADS) {
    const int64_t o = (int64_t)r * p.width + z;
    p.tok[o] = -1;
    p.parent[o] = -1;
    p.cand_id[o] = -1;
  }
  if (j == 0) p.n_rows[r] = n_rows;
}

}  // namespace spec

extern "C" cudaError_t spec_launch_build_tree(int32_t batch, int32_t P, int32_t Kc, const int32_t* anchor,
                                              const int32_t* cand_tok, const float* cand_score,
                                              const int32_t* ng_tok, int32_t Lg, const int32_t* ng_len,
                                              const float* ng_score, const float* ng_adj, int32_t width,
                                              int32_t* tok, int32_t* parent, int32_t* cand_id, int32_t* n_rows,
                                              uint32_t* status, cudaStream_t stream) {
  spec::TreeParams p;
  p.batch = batch;
  p.P = P;
  p.Kc = Kc;
  p.Lg = Lg;
  p.width = width;
  p.anchor = anchor;
  p.cand_tok = cand_tok;
  p.cand_score = cand_score;
  p.ng_tok = ng_tok;
  p.ng_len = ng_len;
  p.ng_score = ng_score;
  p.ng_adj = ng_adj;
  p.tok = tok;
  p.parent = parent;
  p.cand_id = cand_id;
  p.n_rows = n_rows;
  p.status = status;
  spec::build_tree_kernel<<<batch, TB_THREADS, 0, stream>>>(p);
  return cudaGetLastError();
}
