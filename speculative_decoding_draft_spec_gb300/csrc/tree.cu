// tree.cu -- the candidate tree of one block-drafter round.
//
// AdaSpark sec. 2.2 (tree shape; n-gram chains branch from the anchor and from
// each pick), sec. 3.3 (n-gram candidates, Eq. (6)), sec. 3.1 with
// Proposition 1 (best-first order) and Algorithm 1 (the first n-1 nodes of
// the order, laid out depth-first):
//   candidates: 0 the anchor; 1 + i Kc + k the k-th ranked candidate of block
//     position i (k = 0 the pick); pick i hangs from pick i-1 (pick 0 from the
//     anchor), the siblings of position i from the pick's parent, as leaves;
//   n-gram chains, c = 0 from the anchor and c >= 1 from pick c-1, in order: a
//     step equal to a drafter child of the current node marks it agreed
//     (lowest index on duplicates) and moves to it; else a step equal to an
//     n-gram child already there (an earlier chain's) moves to it; else it
//     appends an n-gram node.  The other drafter children of every node a
//     chain passes through are contradicted; agreed wins over contradicted;
//   s: the given drafter score + adj if agreed, else - adj if contradicted; or
//     the n-gram score; clamped to [-80, 80];
//   q_j = e^{s_j} / (1 + sum over the children c of parent(j) of e^{s_c})
//     (children summed in index order), Q_j = the product of q along the path
//     from the anchor, in fp64;
//   order: Q descending, ties to the lower index; the tree: the anchor and the
//     first width-1 candidates, depth-first with children in index order.
//
// GB300 layout: one CTA per request, one thread per candidate (at most 512),
// everything in shared memory.  A step's node depends only on its token path
// from the anchor; with up to 32 chains, eight warps find every step's node at
// once from two tables (where each chain's path leaves the picks, and the
// common-prefix length of every pair of chains), while the other eight warps
// form e^s of every drafter candidate for its three cases (fp64 runs on a
// narrow pipe on this part).  More chains: warp 0 merges depth by depth.  The
// new n-gram nodes are numbered by a block-wide count in the order a
// sequential merge would make them.  A node's children are a known index range
// of drafter candidates plus a list of n-gram nodes in index order, so the
// per-parent sums and the depth-first offsets cost O(children) per node; Q is
// formed by pointer jumping along the parent links, the rank of every
// candidate is a count over all candidates, and the subtree sizes come from
// shared-memory atomics along each path.
#include "common.cuh"

namespace spec {

#define TB_THREADS 512
#define TB_MERGE_WARPS 8  // warps that merge up to 32 chains (named barrier 1)

// the merging warps' own barrier, so that the other warps keep working
__device__ __forceinline__ void merge_bar() {
  asm volatile("bar.sync 1, %0;" ::"n"(32 * TB_MERGE_WARPS) : "memory");
}

struct TreeParams {
  int32_t batch, P, Kc, n_chains, Lg, width;
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

// the lowest-index drafter child c0 .. c0 + Kc - 1 with token x, or -1; the
// first four tokens are loaded together (the merge's chain of steps waits on
// this lookup)
__device__ __forceinline__ int32_t child_with(const int32_t* s_tok, int32_t c0, int32_t Kc, int32_t x) {
  int32_t t[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) t[k] = k < Kc ? s_tok[c0 + k] : 0;
  int32_t node = -1;
#pragma unroll
  for (int k = 3; k >= 0; --k)
    if (k < Kc && t[k] == x) node = c0 + k;
  for (int32_t k = 4; k < Kc && node < 0; ++k)
    if (s_tok[c0 + k] == x) node = c0 + k;
  return node;
}

__global__ void __launch_bounds__(TB_THREADS) build_tree_kernel(TreeParams p) {
  __shared__ int32_t s_tok[TB_THREADS], s_par[TB_THREADS], s_dk[TB_THREADS], s_depth[TB_THREADS];
  __shared__ uint8_t s_agree[TB_THREADS], s_contra[TB_THREADS];
  __shared__ double s_e[TB_THREADS], s_den[TB_THREADS], s_Q[TB_THREADS];
  // e^s of the agreed and contradicted cases, until the denominators and Q take the space
  double* const s_ea = s_den;
  double* const s_ec = s_Q;
  __shared__ int32_t s_size[TB_THREADS];
  __shared__ int32_t s_ngfirst[TB_THREADS], s_ngnext[TB_THREADS];
  __shared__ int32_t s_itok[TB_THREADS], s_ipar[TB_THREADS], s_node[TB_THREADS], s_final[TB_THREADS];
  // the selection and the sibling offsets reuse the chain steps' tokens and parents
  int32_t* const s_sel = s_itok;
  int32_t* const s_before = s_ipar;
  // scratch: the merge's path tables, then the Q pointers
  __shared__ int32_t s_bucket[TB_THREADS], s_bpar[TB_THREADS];
  __shared__ int32_t s_N, s_maxd, s_levels, s_len[TB_THREADS], s_wcnt[TB_THREADS / 32];
  __shared__ double s_eng;
  const int r = blockIdx.x, j = threadIdx.x;
  const int lane = j & 31, warp = j >> 5;
  const int P = p.P, Kc = p.Kc, NC = p.n_chains, Lg = p.Lg;
  const int ND = 1 + P * Kc;  // anchor + drafter candidates
  // every global input of the request, loaded at once: the drafter's block,
  // the chains and the per-request scalars
  if (j < ND) {
    if (j == 0) {
      s_tok[0] = p.anchor[r];
      s_par[0] = -1;
      s_depth[0] = 0;
      s_dk[0] = P > 0 ? 1 : -1;
    } else {
      const int i = (j - 1) / Kc, k = (j - 1) - i * Kc;
      s_tok[j] = p.cand_tok[(int64_t)r * P * Kc + (j - 1)];
      s_par[j] = (i == 0) ? 0 : 1 + (i - 1) * Kc;
      s_depth[j] = i + 1;
      // a pick that is not the last has the next position's candidates as children
      s_dk[j] = (k == 0 && i + 1 < P) ? j + Kc : -1;
    }
  }
  s_agree[j] = 0;
  s_contra[j] = 0;
  s_ngfirst[j] = 0x7FFFFFFF;
  s_ngnext[j] = -1;
  s_size[j] = 0;
  if (j == 0) {
    s_maxd = 0;
    s_levels = 0;
  }
  // chain item j = c Lg + t: the t-th step of chain c
  const int nct = NC * Lg;
  if (j < nct) s_itok[j] = p.ng_tok[(int64_t)r * nct + j];
  int32_t my_gl = 0;
  if (j < NC) {
    my_gl = p.ng_len[(int64_t)r * NC + j];
    if (my_gl < 0 || my_gl > Lg) {
      set_status(p.status, SPEC_DEV_BAD_LENGTH);
      my_gl = 0;
    }
    s_len[j] = my_gl;
  }
  if (NC > 32) {
    __syncthreads();  // s_levels is zero from here on
    if (j < NC) atomicMax(&s_levels, j + my_gl);  // chain c's steps sit at depths c+1 .. c+gl
    __syncthreads();
  } else if (warp >= TB_MERGE_WARPS) {
    // the exponential warps signal that their part of the set-up is written
    // and go on without waiting (they read nothing the others write)
    asm volatile("bar.arrive 2, %0;" ::"n"(TB_THREADS) : "memory");
  } else {
    asm volatile("bar.sync 2, %0;" ::"n"(TB_THREADS) : "memory");
  }
  // the node of every chain step.  A step's node depends only on its token
  // path from the anchor (chain c's path: pick_0 .. pick_{c-1}, then its own
  // tokens): while the path follows the picks it is the next pick; at the first
  // step that leaves them, the lowest-index sibling with that step's token
  // (when that position has candidates), else an n-gram node; below, n-gram
  // nodes.  An n-gram node is shared by every chain whose path is the same up
  // to its depth and is made by the first of them in chain order.  The parent
  // of a step with drafter children has its taken child agreed and the others
  // contradicted.  Provisional ids: drafter nodes their index, n-gram nodes
  // ND + the item that makes them.
  auto path_tok = [&](int c, int k) -> int32_t {  // token k (1-based) of chain c's path
    return k <= c ? s_tok[1 + (k - 1) * Kc] : s_itok[c * Lg + (k - c - 1)];
  };
  // e^s of every drafter candidate for each of its three cases (plain,
  // agreed, contradicted) and of an n-gram node, clamped to [-80, 80]: one
  // exponential per thread, item w = 3 (v - 1) + case, then the n-gram node's
  const double adj = (double)p.ng_adj[r];
  auto ex = [](double x) { return exp(x > 80.0 ? 80.0 : (x < -80.0 ? -80.0 : x)); };
  auto exps = [&](int w0, int step) {
    for (int w = w0; w <= 3 * (ND - 1); w += step) {
      if (w == 3 * (ND - 1)) {
        s_eng = ex((double)p.ng_score[r]);
        continue;
      }
      const int v = 1 + w / 3, cs = w - 3 * (v - 1);
      const double sv = (double)p.cand_score[(int64_t)r * P * Kc + (v - 1)];
      if (cs == 0)
        s_e[v] = ex(sv);
      else if (cs == 1)
        s_ea[v] = ex(sv + adj);
      else
        s_ec[v] = ex(sv - adj);
    }
  };
  if (NC <= 32 && warp < TB_MERGE_WARPS) {
    // up to 32 chains: all steps at once by the first 8 warps (their own
    // barrier), from two tables -- the depth at which each chain's path leaves
    // the picks, and the common-prefix length of every pair of chains (c' < c,
    // pair c (c - 1) / 2 + c') -- while the other warps form the exponentials
    constexpr int MT = 32 * TB_MERGE_WARPS;
    int32_t* const s_leave = s_bpar;  // [NC]
    int32_t* const s_lcp = s_bucket;  // [NC (NC - 1) / 2]
    // warp w takes chains w, w + 8, ...: the depth at which the chain's path
    // leaves the picks, 32 steps per ballot
    for (int c = warp; c < NC; c += TB_MERGE_WARPS) {
      const int len = s_len[c];
      int leave = c + len + 1;  // past the last step: never leaves
      for (int t0 = 0; t0 < len; t0 += 32) {
        const int t = t0 + lane, d = c + t + 1;
        const bool off = t < len && (d > P || s_itok[c * Lg + t] != s_tok[1 + (d - 1) * Kc]);
        const unsigned m = __ballot_sync(0xFFFFFFFFu, off);
        if (m != 0u) {
          leave = c + t0 + __ffs(m);
          break;
        }
      }
      if (lane == 0) s_leave[c] = leave;
    }
    merge_bar();
    // pairs c2 < c (pair c (c - 1) / 2 + c2; warp w takes pairs w, w + 8, ...):
    // both paths follow the picks through depth c2, and chain c's through depth
    // c, so the paths part where chain c2 leaves the picks if that is at or
    // before depth c; otherwise they agree through depth c and part at the
    // first difference of the two chains' own tokens
    const int NP = NC * (NC - 1) / 2;
    for (int pi = warp; pi < NP; pi += TB_MERGE_WARPS) {
      int c = (int)((1.0f + sqrtf(1.0f + 8.0f * (float)pi)) * 0.5f);
      while (c * (c - 1) / 2 > pi) --c;
      while ((c + 1) * c / 2 <= pi) ++c;
      const int c2 = pi - c * (c - 1) / 2;
      const int lim = min(c2 + s_len[c2], c + s_len[c]);
      const int lv = s_leave[c2];
      int lcp = lv <= c ? min(lv - 1, lim) : lim;
      if (lv > c) {
        for (int k0 = c + 1; k0 <= lim; k0 += 32) {
          const int k = k0 + lane;
          const unsigned m = __ballot_sync(
              0xFFFFFFFFu, k <= lim && s_itok[c2 * Lg + (k - c2 - 1)] != s_itok[c * Lg + (k - c - 1)]);
          if (m != 0u) {
            lcp = k0 + __ffs(m) - 2;
            break;
          }
        }
      }
      if (lane == 0) s_lcp[pi] = lcp;
    }
    merge_bar();
    for (int i = j; i < nct; i += MT) {
      const int c = i / Lg, t = i - c * Lg;
      if (t >= s_len[c]) continue;
      const int d = c + t + 1, leave = s_leave[c];
      auto node_at = [&](int dd) -> int32_t {
        if (dd < leave) return 1 + (dd - 1) * Kc;  // the pick at depth dd
        if (dd == leave && dd <= P) {
          const int32_t x = path_tok(c, dd);
          for (int k = 1; k < Kc; ++k)
            if (s_tok[1 + (dd - 1) * Kc + k] == x) return 1 + (dd - 1) * Kc + k;  // a sibling
        }
        int first = c;
        for (int c2 = 0; c2 < c; ++c2)
          if (s_lcp[c * (c - 1) / 2 + c2] >= dd) {
            first = c2;
            break;
          }
        return ND + first * Lg + (dd - first - 1);
      };
      const int32_t node = node_at(d);
      const int32_t par = t == 0 ? (c == 0 ? 0 : 1 + (c - 1) * Kc) : node_at(d - 1);
      s_node[i] = node;
      s_ipar[i] = par;
      const int32_t c0 = par < ND ? s_dk[par] : -1;
      if (c0 >= 0) {
        for (int32_t k = 0; k < Kc; ++k)
          if (c0 + k != node) s_contra[c0 + k] = 1;
        if (node < ND) s_agree[node] = 1;
      }
    }
  } else if (NC <= 32) {
    exps(j - 32 * TB_MERGE_WARPS, TB_THREADS - 32 * TB_MERGE_WARPS);
  } else if (warp == 0) {
    // more than 32 chains: depth by depth by warp 0, 32 chains a round (lane
    // = chain), the first chain with the same (parent, token) at a depth the
    // lowest lane of its __match_any_sync group or an earlier round's chain
    const int levels = s_levels;
    for (int d = 1; d <= levels; ++d) {
      for (int cb = 0; cb < NC; cb += 32) {
        const int c = cb + lane, t = d - c - 1;
        const bool active = c < NC && t >= 0 && t < s_len[c];
        const int jj = c * Lg + t;
        int32_t par = -1, xt = 0, node = -1;
        if (active) {
          par = t == 0 ? (c == 0 ? 0 : 1 + (c - 1) * Kc) : s_node[jj - 1];
          xt = s_itok[jj];
          const int32_t c0 = par < ND ? s_dk[par] : -1;
          if (c0 >= 0) {
            node = child_with(s_tok, c0, Kc, xt);
            for (int32_t k = 0; k < Kc; ++k)
              if (c0 + k != node) s_contra[c0 + k] = 1;
            if (node >= 0) s_agree[node] = 1;
          }
        }
        const bool need = active && node < 0;
        const unsigned mask = __ballot_sync(0xFFFFFFFFu, need);
        if (need) {
          const unsigned long long key = ((unsigned long long)(uint32_t)par << 32) | (uint32_t)xt;
          const unsigned grp = __match_any_sync(mask, key);
          const int c1 = cb + __ffs(grp) - 1;
          node = ND + c1 * Lg + (d - c1 - 1);
          // chains of earlier rounds come first in chain order
          for (int c2 = 0; c2 < cb; ++c2) {
            const int t2 = d - c2 - 1;
            if (t2 < 0 || t2 >= s_len[c2]) continue;
            const int j2 = c2 * Lg + t2;
            if (s_itok[j2] == xt && s_ipar[j2] == par) {
              node = ND + j2;
              break;
            }
          }
        }
        if (active) {
          s_node[jj] = node;
          s_ipar[jj] = par;
        }
        __syncwarp();
      }
    }
  } else {
    exps(j - 32, TB_THREADS - 32);  // meanwhile, by the other warps
  }
  __syncthreads();
  // the n-gram nodes in the order the sequential merge makes them: a step that
  // makes its node gets index ND + (the steps before it, in chain order, that
  // make theirs)
  const int my_c = Lg > 0 ? j / Lg : 0, my_t = Lg > 0 ? j - my_c * Lg : 0;
  const bool item = j < nct && my_t < s_len[my_c];
  const bool makes = item && s_node[j] == ND + j;
  {
    const unsigned bal = __ballot_sync(0xFFFFFFFFu, makes);
    if (lane == 0) s_wcnt[warp] = __popc(bal);
    __syncthreads();
    int32_t before = __popc(bal & ((1u << lane) - 1u)), all = 0;
#pragma unroll
    for (int w = 0; w < TB_THREADS / 32; ++w) {
      before += w < warp ? s_wcnt[w] : 0;
      all += s_wcnt[w];
    }
    if (makes) s_final[j] = ND + before;
    if (j == 0) s_N = ND + all;
  }
  __syncthreads();
  const int N = s_N;
  if (makes) {
    const int32_t v = s_final[j];
    const int32_t par = s_ipar[j];
    const int32_t pv = par < ND ? par : s_final[par - ND];
    s_tok[v] = s_itok[j];
    s_par[v] = pv;
    s_depth[v] = my_c + my_t + 1;
    atomicMin(&s_ngfirst[pv], v);
  }
  if (j < ND) atomicMax(&s_maxd, s_depth[j]);
  if (makes) atomicMax(&s_maxd, my_c + my_t + 1);
  __syncthreads();
  // each n-gram node's next sibling: the smallest larger index among the nodes
  // made at its depth with its parent; e^s of every candidate
  if (makes) {
    const int32_t v = s_final[j], par = s_ipar[j], d = my_c + my_t + 1;
    int32_t nx = 0x7FFFFFFF;
    for (int c2 = 0; c2 < NC; ++c2) {
      const int t2 = d - c2 - 1;
      if (t2 < 0 || t2 >= s_len[c2]) continue;
      const int j2 = c2 * Lg + t2;
      if (s_node[j2] == ND + j2 && s_ipar[j2] == par) {
        const int32_t w = s_final[j2];
        if (w > v && w < nx) nx = w;
      }
    }
    s_ngnext[v] = nx == 0x7FFFFFFF ? -1 : nx;
  }
  if (j < N) {
    if (s_ngfirst[j] == 0x7FFFFFFF) s_ngfirst[j] = -1;
    if (j >= 1 && j < ND)
      s_e[j] = s_agree[j] ? s_ea[j] : (s_contra[j] ? s_ec[j] : s_e[j]);
    else if (j >= ND)
      s_e[j] = s_eng;
  }
  const int32_t maxd = s_maxd;
  __syncthreads();  // every candidate's e^s is chosen
  // Eq. (6) denominators: thread j sums its own children in index order, the
  // drafter range first
  if (j < N) {
    double den = 1.0;
    const int32_t c0 = j < ND ? s_dk[j] : -1;
    if (c0 >= 0)
      for (int32_t k = 0; k < Kc; ++k) den += s_e[c0 + k];
    for (int32_t g = s_ngfirst[j]; g >= 0; g = s_ngnext[g]) den += s_e[g];
    s_den[j] = den;
  }
  __syncthreads();
  // q_j = e^{s_j} / den(parent), then Q_j, the product of q along the path
  // from the anchor, by pointer jumping: after round k a node holds the
  // product of the last 2^k factors of its path and the node 2^k steps up (the
  // anchor holds 1 and points to itself), so max depth d needs ceil(log2 d)
  // rounds.  The products associate differently from the left-to-right
  // definition, which moves Q by a few units in the last place.
  // two buffers each for Q and the jump pointers (the denominators and the
  // merge's table are free by now), so a round needs one barrier
  double* qa = s_Q;
  double* qb = s_den;
  int32_t* ua = s_bucket;
  int32_t* ub = s_bpar;
  if (j < N) {
    qa[j] = j > 0 ? s_e[j] / s_den[s_par[j]] : 1.0;
    ua[j] = j > 0 ? s_par[j] : 0;
  }
  __syncthreads();
  for (int32_t covered = 1; covered < maxd; covered <<= 1) {
    if (j < N) {
      const int32_t u = ua[j];
      qb[j] = qa[u] * qa[j];
      ub[j] = ua[u];
    }
    __syncthreads();
    double* const tq = qa;
    qa = qb;
    qb = tq;
    int32_t* const tu = ua;
    ua = ub;
    ub = tu;
  }
  // best-first rank (Q descending, ties to the lower index) and selection
  if (j < N) {
    bool sel = (j == 0);
    if (j > 0) {
      // Q >= 0, so its bit pattern orders like its value: integer compares
      // (fp64 compares run on the narrow FP64 pipe)
      const unsigned long long kj = (unsigned long long)__double_as_longlong(qa[j]);
      int32_t rank = 0;
#pragma unroll 8
      for (int32_t i = 1; i < N; ++i) {
        const unsigned long long ki = (unsigned long long)__double_as_longlong(qa[i]);
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
    const int32_t c0 = j < ND ? s_dk[j] : -1;
    if (c0 >= 0)
      for (int32_t k = 0; k < Kc; ++k)
        if (s_sel[c0 + k]) {
          s_before[c0 + k] = run;
          run += s_size[c0 + k];
        }
    for (int32_t g = s_ngfirst[j]; g >= 0; g = s_ngnext[g])
      if (s_sel[g]) {
        s_before[g] = run;
        run += s_size[g];
      }
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
                                              const int32_t* ng_tok, int32_t n_chains, int32_t Lg,
                                              const int32_t* ng_len,
                                              const float* ng_score, const float* ng_adj, int32_t width,
                                              int32_t* tok, int32_t* parent, int32_t* cand_id, int32_t* n_rows,
                                              uint32_t* status, cudaStream_t stream) {
  spec::TreeParams p;
  p.batch = batch;
  p.P = P;
  p.Kc = Kc;
  p.n_chains = n_chains;
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
