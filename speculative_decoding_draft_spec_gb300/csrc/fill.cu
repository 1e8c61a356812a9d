// fill.cu -- the n-gram chains of a candidate tree.
//
// AdaSpark sec. 2.2 (n-gram chains branch from the anchor and from each pick
// and may run past the drafter's block) and sec. 3.3 ("N-gram candidates"),
// with the parameter table's three-token follower context and 32-token depth:
// for request r with committed text x = hist[r][0 .. T-1] (its last token the
// anchor), chain c = 0 starts at the anchor and chain c >= 1 at pick c-1, with
// context ctx = x, pick_0 .. pick_{c-1}.  Each step appends one token y:
//   1. reading along an earlier passage whose next position is <= T-1: y is
//      that token;
//   2. else the earlier occurrence of ctx: over end positions j <= T-2,
//      l(j) = common-suffix length of x[..j] and ctx capped at copy_cap and
//      j+1; among l >= n_min the largest (l, j); y = x[j+1] and the chain
//      reads on from j+2;
//   3. else the most frequent follower x[j+1] of the last three tokens of ctx
//      over j in [2, T-2], ties to the follower seen most recently;
//   4. else the chain stops.
// A chain ends at depth max_depth below the anchor (Lg tokens at most).  ev
// holds each token's evidence: the length of the copy it continues (capped at
// copy_cap) for steps 1-2, minus the follower's count for step 3.
//
// GB300 layout: one CTA of 256 threads per (chain, request).  The request's
// text is staged in shared memory once (when it fits: FL_STAGE_MAX tokens),
// so the passes below read on-chip memory instead of making one memory round
// trip per position.  The chain's steps are sequential; a lookup is one
// block-wide pass over the text (each thread tests its end positions four at
// a time, extends the matches it finds, and the block takes the max of
// (l << 32 | j)), a follower step one pass that counts followers in a
// shared-memory hash table (atomics) and one max over it (more passes, over
// halves of the follower value range, where a context has more distinct
// followers than the table holds).  Reading on along a
// passage needs no lookup, so a whole run of such steps is one parallel copy.
// All threads carry the same chain state, so every branch is block-uniform.
#include "common.cuh"

namespace spec {

#define FL_THREADS 256
#define FL_HASH 2048  // follower table entries (a power of two)
#define FL_STAGE_MAX 16384  // longest text staged in shared memory (64 KB)
#define FL_RANGES 40        // follower ranges pending at once (21 splits deep at most)

struct FillParams {
  const int32_t* hist;
  int64_t stride;
  const int32_t* hist_len;
  int32_t P, Kc;
  const int32_t* cand_tok;
  int32_t n_min, copy_cap, max_depth, Lg;
  int32_t stage;  // the texts are staged in shared memory (stride <= FL_STAGE_MAX)
  int32_t* ng_tok;
  int32_t* ng_len;
  int32_t* ng_ev;
  uint32_t* status;
};

__device__ __forceinline__ unsigned long long block_max_u64(unsigned long long v, unsigned long long* s_red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long t = __shfl_xor_sync(0xFFFFFFFFu, v, o);
    v = t > v ? t : v;
  }
  if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = v;
  __syncthreads();
  unsigned long long m = 0;
#pragma unroll
  for (int w = 0; w < FL_THREADS / 32; ++w) m = s_red[w] > m ? s_red[w] : m;
  return m;
}

__global__ void __launch_bounds__(FL_THREADS) ngram_fill_kernel(FillParams p) {
  // [stride] the staged text (when p.stage), then [P + Lg + 1]: the picks on
  // the path, then the chain
  extern __shared__ __align__(16) int32_t s_dyn[];
  __shared__ unsigned long long s_key[FL_HASH];  // (1 << 32) | follower, 0 = empty
  __shared__ int32_t s_cnt[FL_HASH], s_last[FL_HASH];
  __shared__ unsigned long long s_red[FL_THREADS / 32];
  __shared__ int32_t s_overflow;
  // the follower value ranges still to count, [s_rlo, s_rhi) (a stack)
  __shared__ unsigned long long s_rlo[FL_RANGES], s_rhi[FL_RANGES];
  __shared__ int32_t s_sp;
  const int tid = threadIdx.x;
  const int c = blockIdx.x, r = blockIdx.y;
  const int C = p.P + 1;
  const int32_t* x = p.hist + (int64_t)r * p.stride;
  int32_t T = p.hist_len[r];
  if (T < 0 || (int64_t)T > p.stride) {
    if (tid == 0 && c == 0) set_status(p.status, SPEC_DEV_BAD_LENGTH);
    T = 0;
  }
  int32_t cap = p.max_depth - c;
  if (cap > p.Lg) cap = p.Lg;
  if (T < 1 || cap < 0) cap = 0;  // no anchor
  int32_t* const s_x = s_dyn;
  int32_t* const s_ext = s_dyn + (p.stage ? ((p.stride + 3) & ~3) : 0);
  if (p.stage && cap > 0) {
    // the text, four tokens per load where the row allows it
    if ((p.stride & 3) == 0 && (reinterpret_cast<uintptr_t>(x) & 15u) == 0) {
      const int4* x4 = reinterpret_cast<const int4*>(x);
      for (int i = tid; 4 * i < T; i += FL_THREADS) reinterpret_cast<int4*>(s_x)[i] = __ldg(x4 + i);
    } else {
      for (int i = tid; i < T; i += FL_THREADS) s_x[i] = __ldg(x + i);
    }
  }
  const int32_t* const xs = p.stage ? s_x : x;  // the text, staged or in memory
  for (int i = tid; i < c; i += FL_THREADS) s_ext[i] = p.cand_tok[((int64_t)r * p.P + i) * p.Kc];
  if (tid == 0) s_overflow = 0;
  int32_t* out = p.ng_tok + ((int64_t)r * C + c) * p.Lg;
  int32_t* ev = p.ng_ev + ((int64_t)r * C + c) * p.Lg;
  __syncthreads();
  // ctx = x ++ s_ext[0 .. m-1]
  auto ctx = [&](int64_t i) -> int32_t { return i < T ? xs[i] : s_ext[i - T]; };
  int32_t m = c, n = 0;
  int64_t q = -1;            // the passage's next position in x, or -1
  int32_t run = 0;           // the length of the copy being continued
  while (n < cap) {
    int32_t y = -1, e = 0;
    bool found = false;
    if (q >= 0 && q <= T - 1) {
      // reading along the passage needs no lookup: the next k tokens of the
      // text at once, each with the copy length it continues
      const int32_t k = (int32_t)min((int64_t)(cap - n), (int64_t)T - q);
      for (int i = tid; i < k; i += FL_THREADS) {
        const int32_t t = xs[q + i];
        out[n + i] = t;
        ev[n + i] = min(run + 1 + i, p.copy_cap);
        s_ext[m + i] = t;
      }
      n += k;
      m += k;
      q += k;
      run = min(run + k, p.copy_cap);
      __syncthreads();  // the new tokens are visible to every thread's ctx
      continue;
    } else {
      // the earlier occurrence of ctx: the largest (l, j)
      const int64_t len = (int64_t)T + m;
      const int32_t last = ctx(len - 1);
      unsigned long long best = 0;
      for (int64_t j0 = tid; j0 <= (int64_t)T - 2; j0 += 4 * FL_THREADS) {
        int32_t v[4];  // four end positions' tokens, loaded together
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int64_t j = j0 + u * FL_THREADS;
          v[u] = j <= (int64_t)T - 2 ? xs[j] : ~last;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (v[u] != last) continue;
          const int64_t j = j0 + u * FL_THREADS;
          const int32_t lim = (int32_t)min((int64_t)p.copy_cap, j + 1);
          int32_t l = 1;
          while (l < lim && xs[j - l] == ctx(len - 1 - l)) ++l;
          if (l >= p.n_min) {
            const unsigned long long k = ((unsigned long long)l << 32) | (unsigned long long)j;
            best = k > best ? k : best;
          }
        }
      }
      best = block_max_u64(best, s_red);
      if (best != 0ull) {
        const int64_t j = (int64_t)(uint32_t)best;
        y = xs[j + 1];
        q = j + 2;
        run = (int32_t)(best >> 32);
        e = run;
        found = true;
      } else if (len >= 3) {
        // the most frequent follower of the last three tokens, counted in a
        // shared-memory hash table.  When a pass meets more distinct followers
        // than the table holds, the follower value range of that pass is split
        // in halves and each half is counted by a pass of its own; a range of
        // at most FL_HASH values always fits, so the count is exact for any
        // text (at most 21 levels of splitting).  Each follower lives in one
        // range, so the best (count, last position) over the ranges is the
        // best overall.
        const int32_t a = ctx(len - 3), b = ctx(len - 2), d = last;
        unsigned long long top = 0;
        if (tid == 0) {
          s_rlo[0] = 0ull;
          s_rhi[0] = 1ull << 32;
          s_sp = 1;
        }
        __syncthreads();
        while (s_sp > 0) {  // block-uniform: s_sp changes only between barriers
          const unsigned long long lo = s_rlo[s_sp - 1], hi = s_rhi[s_sp - 1];
          for (int h = tid; h < FL_HASH; h += FL_THREADS) {
            s_key[h] = 0ull;
            s_cnt[h] = 0;
            s_last[h] = -1;
          }
          if (tid == 0) s_overflow = 0;
          __syncthreads();
          for (int64_t j = 2 + tid; j <= (int64_t)T - 2; j += FL_THREADS) {
            if (xs[j] != d || xs[j - 1] != b || xs[j - 2] != a) continue;
            const int32_t f = xs[j + 1];
            if ((unsigned long long)(uint32_t)f < lo || (unsigned long long)(uint32_t)f >= hi) continue;
            const unsigned long long key = (1ull << 32) | (unsigned long long)(uint32_t)f;
            uint32_t h = ((uint32_t)f * 2654435761u) >> (32 - 11);
            bool placed = false;
            for (int probe = 0; probe < FL_HASH && !placed; ++probe) {
              const unsigned long long prev = atomicCAS(&s_key[h], 0ull, key);
              if (prev == 0ull || prev == key) {
                atomicAdd(&s_cnt[h], 1);
                atomicMax(&s_last[h], (int32_t)j);
                placed = true;
              }
              h = (h + 1) & (FL_HASH - 1);
            }
            if (!placed) s_overflow = 1;
          }
          __syncthreads();
          if (s_overflow) {
            __syncthreads();  // every thread has read s_overflow and the range
            if (tid == 0) {   // replace the range by its halves, the lower on top
              const unsigned long long mid = lo + (hi - lo) / 2;
              s_rlo[s_sp - 1] = mid;
              s_rhi[s_sp - 1] = hi;
              s_rlo[s_sp] = lo;
              s_rhi[s_sp] = mid;
              ++s_sp;
            }
            __syncthreads();
            continue;
          }
          unsigned long long best_here = 0;
          for (int h = tid; h < FL_HASH; h += FL_THREADS)
            if (s_key[h] != 0ull) {
              const unsigned long long k = ((unsigned long long)s_cnt[h] << 32) | (unsigned long long)s_last[h];
              best_here = k > best_here ? k : best_here;
            }
          best_here = block_max_u64(best_here, s_red);
          top = best_here > top ? best_here : top;
          __syncthreads();  // every thread has read s_sp and s_red
          if (tid == 0) --s_sp;
          __syncthreads();
        }
        if (top != 0ull) {
          y = xs[(int64_t)(uint32_t)top + 1];
          e = -(int32_t)(top >> 32);
          q = -1;
          run = 0;
          found = true;
        }
      }
    }
    if (!found) break;
    if (tid == 0) {
      out[n] = y;
      ev[n] = e;
      s_ext[m] = y;
    }
    ++n;
    ++m;
    __syncthreads();  // the new token is visible to every thread's ctx
  }
  for (int k = n + tid; k < p.Lg; k += FL_THREADS) {
    out[k] = -1;
    ev[k] = 0;
  }
  if (tid == 0) p.ng_len[(int64_t)r * C + c] = n;
}

}  // namespace spec

extern "C" cudaError_t spec_launch_ngram_fill(const int32_t* hist, int64_t hist_stride, const int32_t* hist_len,
                                              int32_t batch, int32_t P, int32_t Kc, const int32_t* cand_tok,
                                              int32_t n_min, int32_t copy_cap, int32_t max_depth, int32_t Lg,
                                              int32_t* ng_tok, int32_t* ng_len, int32_t* ng_ev, uint32_t* status,
                                              cudaStream_t stream) {
  spec::FillParams fp;
  fp.hist = hist;
  fp.stride = hist_stride;
  fp.hist_len = hist_len;
  fp.P = P;
  fp.Kc = Kc;
  fp.cand_tok = cand_tok;
  fp.n_min = n_min;
  fp.copy_cap = copy_cap;
  fp.max_depth = max_depth;
  fp.Lg = Lg;
  fp.ng_tok = ng_tok;
  fp.ng_len = ng_len;
  fp.ng_ev = ng_ev;
  fp.status = status;
  fp.stage = hist_stride <= FL_STAGE_MAX ? 1 : 0;
  const size_t smem =
      ((fp.stage ? (size_t)((hist_stride + 3) & ~(int64_t)3) : 0) + (size_t)(P + Lg + 1)) * sizeof(int32_t);
  cudaError_t e = cudaFuncSetAttribute(spec::ngram_fill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  spec::ngram_fill_kernel<<<dim3(P + 1, batch), FL_THREADS, smem, stream>>>(fp);
  return cudaGetLastError();
}
