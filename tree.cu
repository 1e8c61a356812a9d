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
// everything in shared memory.  Thread 0 merges the n-gram chain (a short
// sequential walk).  The per-parent sums, the rank of every candidate (a count
// over all candidates) and the depth-first positions (subtree sizes by
// shared-memory atomics, then a sum along the path) are thread-parallel; Q is
// formed level by level from the anchor, one barrier per tree level.
#include "common.cuh"
static __device__ unsigned long long g_t[64][16];
__device__ __forceinline__ unsigned long long gt_() { unsigned long long t; asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t)); return t; }

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
  __shared__ int32_t s_depth[TB_THREADS];
  __shared__ int32_t s_N, s_maxd;
  const int r = blockIdx.x, j = threadIdx.x;
  const int P = p.P, Kc = p.Kc;
  const int ND = 1 + P * Kc;  // anchor + drafter candidates
  // the drafter's block
  if (threadIdx.x == 0 && blockIdx.x < 64) g_t[blockIdx.x][0] = gt_();
  if (j < ND) {
    if (j == 0) {
      s_tok[0] = p.anchor[r];
      s_par[0] = -1;
    } else {
      const int i = (j - 1) / Kc;
      s_tok[j] = p.cand_tok[(int64_t)r * P * Kc + (j - 1)];
      s_par[j] = (i == 0) ? 0 : 1 + (i - 1) * Kc;
    }
    s_flag[j] = 0;
  }
  s_size[j] = 0;
  if (j == 0) s_maxd = 0;
  __syncthreads();
  // the n-gram chain from the anchor  if (threadIdx.x == 0 && blockIdx.x < 64) g_t[blockIdx.x][1] = gt_();
 (sequential by definition: each step
  // depends on where the previous one went)
  if (j == 0) {
    int32_t gl = p.ng_len[r];
    if (gl < 0 || gl > p.Lg) {
      set_status(p.status, SPEC_DEV_BAD_LENGTH);
      gl = 0;
    }
    int32_t cur = 0, N = ND;
    for (int32_t t = 0; t < gl; ++t) {
      const int32_t x = p.ng_tok[(int64_t)r * p.Lg + t];
      // the drafter children of cur: position 0's candidates under the anchor,
      // position i+1's under pick i; none under a sibling or an n-gram node
      int32_t c0 = 0, c1 = 0;
      if (cur == 0) {
        c0 = 1;
        c1 = (P > 0) ? 1 + Kc : 1;
      } else if (cur < ND && (cur - 1) % Kc == 0 && (cur - 1) / Kc + 1 < P) {
        c0 = cur + Kc;  // 1 + (i + 1) Kc
        c1 = c0 + Kc;
      }
      int32_t hit = -1;
      for (int32_t c = c0; c < c1; ++c)
        if (s_tok[c] == x) {
          hit = c;
          break;
        }
      for (int32_t c = c0; c < c1; ++c)
        if (c != hit) s_flag[c] = -1;
      if (hit >= 0) {
        s_flag[hit] = 1;
        cur = hit;
      } else {
        s_tok[N] = x;
        s_par[N] = cur;
        s_flag[N] = 0;
        cur = N;
        ++N;
      }
    }
    s_N = N;
  }
  __syncthreads();
  const int N = s_N;
  if (threadIdx.x == 0 && blockIdx.x < 64) g_t[blockIdx.x][2] = gt_();
  // scores and e^s
  if (j >= 1 && j < N) {
    double s;
    if (j < ND) {
      const double adj = (double)p.ng_adj[r];
      s = (double)p.cand_score[(int64_t)r * P * Kc + (j - 1)];
      s += (s_flag[j] > 0 ? adj : 0.0) - (s_flag[j] < 0 ? adj : 0.0);
    } else {
      s = (double)p.ng_score[r];
    }
    s = s > 80.0 ? 80.0 : (s < -80.0 ? -80.0 : s);
    s_e[j] = exp(s);
  }
  __syncthreads();
  // Eq. (6) denominators  if (threadIdx.x == 0 && blockIdx.x < 64) g_t[blockIdx.x][3] = gt_();
: thread j sums its own children in index order
  if (j < N) {
    double den = 1.0;
    for (int32_t c = j + 1; c < N; ++c)
      if (s_par[c] == j) den += s_e[c];
    s_den[j] = den;
  }
  __syncthreads();
  // depths, then Q_j  if (threadIdx.x == 0 && blockIdx.x < 64) g_t[blockIdx.x][4] = gt_();
 = Q_parent(j) q_j level by level from the anchor down
  // (the order of the definition's products)
  if (j < N) {
    int32_t d = 0;
    for (int32_t a = j; a != 0; a = s_par[a]) ++d;
    s_depth[j] = d;
    atomicMax(&s_maxd, d);
  }
  if (j == 0) s_Q[0] = 1.0;
  __syncthreads();
  const int32_t maxd = s_maxd;
  if (threadIdx.x == 0 && blockIdx.x < 64) g_t[blockIdx.x][5] = gt_();
  for (int32_t d = 1; d <= maxd; ++d) {
    if (j < N && s_depth[j] == d) {
      const int32_t a = s_par[j];
      s_Q[j] = s_Q[a] * (s_e[j] / s_den[a]);
    }
    __syncthreads();
  }
  // best-first rank  if (threadIdx.x == 0 && blockIdx.x < 64) g_t[blockIdx.x][6] = gt_();
 (Q descending, ties to the lower index) and selection
  if (j < N) {
    bool sel = (j == 0);
    if (j > 0) {
      const double Qj = s_Q[j];
      int32_t rank = 0;
      for (int32_t i = 1; i < N; ++i) {
        const double Qi = s_Q[i];
        rank += (Qi > Qj || (Qi == Qj && i < j)) ? 1 : 0;
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
  // before[c]:  if (threadIdx.x == 0 && blockIdx.x < 64) g_t[blockIdx.x][7] = gt_();
 the rows that the selected earlier siblings of c occupy
  if (j < N && s_sel[j]) {
    int32_t run = 0;
    for (int32_t c = j + 1; c < N; ++c)
      if (s_par[c] == j && s_sel[c]) {
        s_before[c] = run;
        run += s_size[c];
      }
  }
  __syncthreads();
  // depth-first position:  if (threadIdx.x == 0 && blockIdx.x < 64) g_t[blockIdx.x][8] = gt_();
 one row per ancestor step, plus the earlier
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
  if (threadIdx.x == 0 && blockIdx.x < 64) g_t[blockIdx.x][9] = gt_();
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

extern "C" int tphase_get(unsigned long long* o) { return (int)cudaMemcpyFromSymbol(o, g_t, sizeof(unsigned long long) * 64 * 16); }
