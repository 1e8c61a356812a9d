// ngram.cu -- step 1 of the round: n-gram prompt lookup (and, fused with it,
// step 2 in spec_draft_and_price).
//
// Hybrid Spark sec. 4.1: the n-gram drafter proposes up to L tokens following
// the longest earlier occurrence of the request's last n_min..n_max tokens
// (sec. 5.1: the longest match is the one used); sec. 4.2 defines the features
// n (match length), a (runner-up agreement) and m (copy length, capped).
// Every earlier end position j <= T-2 has a match length l(j), the
// common-suffix length of x[..j] and x[..T-1] capped at copy_cap; candidates
// (l(j) >= n_min) rank by (l(j), j) descending.
//
// GB300 layout: one CTA per request, or one thread-block cluster per request
// for histories over 8192 tokens.  A cluster's CTAs split the candidate
// positions into contiguous chunks; each CTA stages its chunk (plus a copy_cap
// halo behind it) and the request's last copy_cap tokens into shared memory
// with one-dimensional bulk async copies completed on an mbarrier (bounded
// wait).  Candidates are found four positions per 16-byte shared-memory load
// (with n_min >= 2 they must also match the second-to-last token); match
// lengths up to 8 come from independent compares against the suffix held in
// registers, and longer matches are queued and extended by the whole warp,
// 32 positions per ballot.  A top-2 of packed (l, j) keys is reduced with
// warp shuffles; cluster rank 0 merges the CTAs' top-2 through distributed
// shared memory and writes the proposal and features.
#include <cooperative_groups.h>

#include "pricing.cuh"

namespace cg = cooperative_groups;

namespace spec {

struct NgramParams {
  const int32_t* hist;
  int64_t stride;
  const int32_t* hist_len;
  int32_t batch, n_min, n_max, L, cap;
  int32_t* g;
  int32_t* g_len;
  int32_t* match_n;
  int32_t* agree;
  int32_t* copy_len;
  uint32_t* status;
  int32_t win_cap;  // tokens of the staged window per CTA (multiple of 4)
  int32_t suf_cap;  // tokens of the staged suffix (multiple of 4)
  int32_t use_bulk; // 1: history rows are 16-byte aligned (bulk copies allowed)
  // fused pricing (draft-and-price kernel only)
  const int32_t* d;
  const float* c;
  const int32_t* d_len;
  PriceCtx cx;
  SelectCtx sc;
  uint32_t* arrive;  // request arrival counter (zero between calls)
  // batches of at most SPEC_PACKED_ARRIVAL requests: request r adds (its valid
  // slots + 1) << (SPEC_PACKED_BITS r) here instead (zero between calls), so the last arrival
  // returns every request's count with the arrival itself
  unsigned long long* arrive64;
  // the Eq. (1) table staged in the pricing CTA's shared memory: its offset in
  // 4-byte words (16-byte aligned), -1 when it is read from global memory
  int32_t tab_off;
  uint32_t tab_bytes;
};

// top-2 of a set of distinct keys held as (b1 >= b2) per lane, merged across the warp
__device__ __forceinline__ void warp_top2(unsigned long long& b1, unsigned long long& b2) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long o1 = __shfl_xor_sync(0xFFFFFFFFu, b1, o);
    const unsigned long long o2 = __shfl_xor_sync(0xFFFFFFFFu, b2, o);
    if (b1 > o1) {
      b2 = b2 > o1 ? b2 : o1;
    } else {
      b2 = b1 > o2 ? b1 : o2;
      b1 = o1;
    }
  }
}

__device__ __forceinline__ void top2_insert(unsigned long long& b1, unsigned long long& b2,
                                            unsigned long long k) {
  if (k > b1) {
    b2 = b1;
    b1 = k;
  } else if (k > b2) {
    b2 = k;
  }
}

#define NG_SHORT 8  // tokens a thread extends a candidate by itself
#define NG_QCAP 64  // queued long candidates per warp
#define NG_UNROLL 4 // 16-byte groups per thread in flight in the candidate filter
#define SPEC_PACKED_ARRIVAL 10  // batches whose per-request counts ride in one 64-bit arrival word
#define SPEC_PACKED_BITS 6      // bits per request: valid slots + 1 <= SPEC_MAX_L + 1 = 32 < 2^6

// device-scope 64-bit fetch-add with acquire-release ordering
__device__ __forceinline__ unsigned long long atomic_add_acq_rel_u64(unsigned long long* p, unsigned long long v) {
  unsigned long long old;
  asm volatile("atom.add.acq_rel.gpu.u64 %0, [%1], %2;" : "=l"(old) : "l"(p), "l"(v) : "memory");
  return old;
}

template <bool CLUSTER, bool PRICE>
__global__ void __launch_bounds__(SPEC_CTA_THREADS, 1) ngram_kernel(NgramParams p) {
  extern __shared__ __align__(16) int32_t smem_tok[];
  __shared__ __align__(8) uint64_t bar;
  __shared__ unsigned long long warp_best[SPEC_WARPS_PER_CTA][2];
  __shared__ unsigned long long cta_best[2];
  __shared__ int32_t s_flag;

  cg::cluster_group cluster = cg::this_cluster();
  const int C = CLUSTER ? (int)cluster.num_blocks() : 1;
  const int rank = CLUSTER ? (int)cluster.block_rank() : 0;
  const int r = blockIdx.x / C;
  const int tid = threadIdx.x;
  const int32_t* x = p.hist + (int64_t)r * p.stride;
  // one CTA per request (rows of at most 8192 tokens): the whole row is copied
  // at once, before its length is read, so the copy and that load overlap
  const bool whole_row = !CLUSTER && p.use_bulk;
  // fused pricing: the CTA that prices (rank 0) copies the Eq. (1) table into
  // its shared memory behind the history, so the row the scan picks is an
  // on-chip read when the pricing needs it
  __shared__ __align__(8) uint64_t tbar;
  const bool tab_smem = PRICE && rank == 0 && p.tab_off >= 0;
  if (tid == 0 && (whole_row || tab_smem)) {
    if (whole_row) mbar_init(&bar, 1);
    if (tab_smem) mbar_init(&tbar, 1);
    fence_mbar_init();
    if (whole_row) {
      mbar_arrive_expect_tx(&bar, (uint32_t)p.stride * 4u);
      bulk_g2s(smem_tok, x, (uint32_t)p.stride * 4u, &bar);
    }
    if (tab_smem) {
      mbar_arrive_expect_tx(&tbar, p.tab_bytes);
      bulk_g2s(smem_tok + p.tab_off, p.cx.table, p.tab_bytes, &tbar);
    }
  }

  const int32_t T = p.hist_len[r];
  const bool valid = (T >= 0) && ((int64_t)T <= p.stride);
  // fused pricing: warp 0 of rank 0 fetches the model drafter's chain now, while
  // the history copy is in flight
  __shared__ PriceStage s_ps;
  __shared__ int32_t s_dl;
  if (PRICE && rank == 0 && tid < 32) {
    if (tid == 0) s_dl = p.d_len[r];
    if (tid < p.cx.K) {
      s_ps.d[tid] = p.d[(int64_t)r * p.cx.K + tid];
      s_ps.c[tid] = p.c[(int64_t)r * p.cx.K + tid];
    }
  }
  // the Eq. (1) table is read once per request after the scan, at a row the scan
  // picks: every CTA brings its share of the table's lines into L2 now, while
  // the history copies are in flight, so that read hits L2
  if (PRICE && !p.cx.tab_const && p.tab_off < 0 && tid < 32) {
    const int64_t n_h = (int64_t)p.cx.L * (SPEC_TAB_N * 2 + 2 * (p.cx.m_cap + 1));  // table floats
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(p.cx.table) & ~(uintptr_t)127;
    const uintptr_t a1 = reinterpret_cast<uintptr_t>(p.cx.table + n_h);
    const uintptr_t step = (uintptr_t)gridDim.x * 32u * 128u;  // one 128-byte line per lane
    for (uintptr_t a = a0 + ((uintptr_t)blockIdx.x * 32u + (uintptr_t)tid) * 128u; a < a1; a += step)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
  }
  const int32_t nc = valid && T >= 2 ? T - 1 : 0;  // candidate end positions 0..T-2
  const int32_t per = (nc + C - 1) / C;
  const int32_t j0 = min(nc, rank * per);
  const int32_t j1 = min(nc, j0 + per);
  const bool work = j0 < j1;

  // staged ranges, rounded to 4-token (16-byte) boundaries (the whole row: both are it)
  const int32_t w0 = whole_row ? 0 : max(0, j0 - p.cap + 1) & ~3;
  const int32_t w1 = whole_row ? (int32_t)p.stride : (j1 + 3) & ~3;
  const int32_t s0 = whole_row ? 0 : max(0, T - p.cap) & ~3;
  const int32_t s1 = whole_row ? (int32_t)p.stride : (T + 3) & ~3;
  int32_t* win = smem_tok;                                   // x[w0 .. w1)
  int32_t* suf = whole_row ? smem_tok : smem_tok + p.win_cap;  // x[s0 .. s1)

  __shared__ int32_t s_q[SPEC_WARPS_PER_CTA][NG_QCAP];  // queued long candidates per warp
  __shared__ int32_t s_qn[SPEC_WARPS_PER_CTA];
  if (tid == 0) s_flag = 0;
  if (tid < SPEC_WARPS_PER_CTA) s_qn[tid] = 0;
  if (whole_row) {
    __syncthreads();  // the barrier's initialisation and s_flag are visible
    if (!mbar_wait_bounded(&bar, 0, 1u << 22)) {
      // the copy has not landed: record it, wait (bounded) for it to finish
      // writing this CTA's shared memory, and skip the scan
      if (tid == 0) set_status(p.status, SPEC_DEV_TIMEOUT);
      atomicOr(&s_flag, 1);
      mbar_wait_bounded(&bar, 0, 1u << 22);
    }
  } else if (work) {
    if (p.use_bulk) {
      if (tid == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
      }
      __syncthreads();
      if (tid == 0) {
        const uint32_t wb = (uint32_t)(w1 - w0) * 4u, sb = (uint32_t)(s1 - s0) * 4u;
        mbar_arrive_expect_tx(&bar, wb + sb);
        bulk_g2s(win, x + w0, wb, &bar);
        bulk_g2s(suf, x + s0, sb, &bar);
      }
      if (!mbar_wait_bounded(&bar, 0, 1u << 22)) {
        // the copy has not landed: record it, wait (bounded) for it to finish
        // writing this CTA's shared memory, and skip the scan
        if (tid == 0) set_status(p.status, SPEC_DEV_TIMEOUT);
        atomicOr(&s_flag, 1);
        mbar_wait_bounded(&bar, 0, 1u << 22);
      }
    } else {
      for (int32_t t = w0 + tid; t < w1; t += blockDim.x) win[t - w0] = t < T ? x[t] : 0;
      for (int32_t t = s0 + tid; t < s1; t += blockDim.x) suf[t - s0] = t < T ? x[t] : 0;
    }
  }
  __syncthreads();

  // Each thread extends its candidates up to NG_SHORT tokens; one still
  // matching there goes to its warp's queue, and the warp then extends the
  // queued candidates 32 positions per step (one ballot per step), so a long
  // copy costs l / 32 steps instead of l dependent compares.
  const int warp = tid >> 5, lane = tid & 31;
  unsigned long long b1 = 0ull, b2 = 0ull;  // packed (l << 32 | j); 0 = none
  if (work && s_flag == 0) {
    const int32_t* wv = win - w0;  // wv[t] = x[t]
    const int32_t* sv = suf - s0;
    // the suffix's last NG_SHORT tokens in registers (entries past the
    // staged suffix are never compared: k < lim <= min(cap, T - 1))
    int32_t sk[NG_SHORT];
#pragma unroll
    for (int k = 0; k < NG_SHORT; ++k) sk[k] = (k < p.cap && k < T) ? sv[T - 1 - k] : 0;
    const int32_t last = sk[0];
    // l(j) up to NG_SHORT by independent compares; a candidate still matching
    // there is queued for its warp (or, with the queue full, extended alone)
    auto extend = [&](int32_t j) {
      const int32_t lim = min(p.cap, j + 1);
      uint32_t ok = 0u;
#pragma unroll
      for (int k = 1; k < NG_SHORT; ++k) ok |= (uint32_t)(k < lim && wv[j - k] == sk[k]) << (k - 1);
      int32_t l = __ffs(~ok);  // the first k that fails, or NG_SHORT
      if (l == NG_SHORT && l < lim) {
        const int slot = atomicAdd(&s_qn[warp], 1);
        if (slot < NG_QCAP) {
          s_q[warp][slot] = j;
          return;
        }
        while (l < lim && wv[j - l] == sv[T - 1 - l]) ++l;
      }
      if (l >= p.n_min) top2_insert(b1, b2, ((unsigned long long)l << 32) | (uint32_t)j);
    };
    // a candidate that also matches the second-to-last token (j >= 1, cap >=
    // 2) is extended; one that does not has l = 1 exactly, so it needs no
    // extension: with n_min = 1 it enters the top two as (1, j), with n_min >= 2
    // it is dropped
    const bool two_ok = p.cap >= 2 && T >= 2;
    const int32_t s1 = two_ok ? sk[1] : 0;
    const bool keep_ones = p.n_min <= 1;
    {
      // candidate filter on 16-byte groups: thread t reads groups t, t + 256, ...
      // (consecutive lanes, consecutive 16 bytes), NG_UNROLL groups in flight;
      // wv is 16-byte aligned at multiples of 4 (the staged window starts at
      // w0 = 0 mod 4 and holds x[w0, w1), w1 = j1 rounded up to 4)
      const int32_t jb = j0 & ~3;
      const int32_t gstride = 4 * (int32_t)blockDim.x;
      for (int32_t c0 = jb + 4 * tid; c0 < j1; c0 += NG_UNROLL * gstride) {
        int4 v[NG_UNROLL];
        int32_t prev[NG_UNROLL];  // x[c - 1], read only when position c is in range
#pragma unroll
        for (int u = 0; u < NG_UNROLL; ++u) {
          const int32_t c = c0 + u * gstride;
          v[u] = c < j1 ? *reinterpret_cast<const int4*>(wv + c) : make_int4(0, 0, 0, 0);
          prev[u] = (two_ok && c < j1 && c >= j0 && c >= 1) ? wv[c - 1] : 0;
        }
        // the groups' match masks, packed four bits per group (bit 4 u + e:
        // position c0 + u gstride + e), so that one copy of the extension code
        // serves every group
        uint32_t ones = 0u, twos = 0u;
#pragma unroll
        for (int u = 0; u < NG_UNROLL; ++u) {
          const int32_t c = c0 + u * gstride;
          uint32_t m = (uint32_t)(v[u].x == last) | ((uint32_t)(v[u].y == last) << 1) |
                       ((uint32_t)(v[u].z == last) << 2) | ((uint32_t)(v[u].w == last) << 3);
          if (c < j0) m &= 0xFu << (j0 - c);                 // before this CTA's range
          if (c + 4 > j1) m &= (1u << max(0, j1 - c)) - 1u;  // past it
          const uint32_t m2 =
              two_ok ? m & ((uint32_t)(prev[u] == s1 && c >= 1) | ((uint32_t)(v[u].x == s1) << 1) |
                            ((uint32_t)(v[u].y == s1) << 2) | ((uint32_t)(v[u].z == s1) << 3))
                     : 0u;
          ones |= (m & ~m2) << (4 * u);
          twos |= m2 << (4 * u);
        }
        // single matches (l = 1) enter the top two as (1, j): no extension
        if (keep_ones) {
          while (ones) {
            const int e = __ffs(ones) - 1;
            ones &= ones - 1u;
            top2_insert(b1, b2, (1ull << 32) | (uint32_t)(c0 + (e >> 2) * gstride + (e & 3)));
          }
        }
        while (twos) {
          const int e = __ffs(twos) - 1;
          twos &= twos - 1u;
          extend(c0 + (e >> 2) * gstride + (e & 3));
        }
      }
    }
    __syncwarp();
    const int nq = min(s_qn[warp], NG_QCAP);
    for (int i = 0; i < nq; ++i) {
      const int32_t j = s_q[warp][i];
      const int32_t lim = min(p.cap, j + 1);
      int32_t l = NG_SHORT;
      while (l < lim) {
        const int32_t t = l + lane;
        const bool ok = t < lim && wv[j - t] == sv[T - 1 - t];
        const uint32_t bad = __ballot_sync(0xFFFFFFFFu, !ok);
        if (bad) {
          l += __ffs(bad) - 1;
          break;
        }
        l += 32;
      }
      if (lane == 0 && l >= p.n_min) top2_insert(b1, b2, ((unsigned long long)l << 32) | (uint32_t)j);
    }
  }
  warp_top2(b1, b2);
  if (lane == 0) {
    warp_best[warp][0] = b1;
    warp_best[warp][1] = b2;
  }
  __syncthreads();
  if (tid == 0) {
    unsigned long long c1 = 0ull, c2 = 0ull;
    for (int w = 0; w < SPEC_WARPS_PER_CTA; ++w) {
      top2_insert(c1, c2, warp_best[w][0]);
      top2_insert(c1, c2, warp_best[w][1]);
    }
    cta_best[0] = c1;
    cta_best[1] = c2;
  }
  if (CLUSTER)
    cluster.sync();
  else
    __syncthreads();

  if (rank == 0) {
    __shared__ unsigned long long fin[2];
    if (tid == 0) {
      unsigned long long c1 = 0ull, c2 = 0ull;
      if (CLUSTER) {
        for (int q = 0; q < C; ++q) {
          const unsigned long long* peer = cluster.map_shared_rank(cta_best, q);
          top2_insert(c1, c2, peer[0]);
          top2_insert(c1, c2, peer[1]);
        }
      } else {
        c1 = cta_best[0];
        c2 = cta_best[1];
      }
      fin[0] = c1;
      fin[1] = c2;
      if (!valid) set_status(p.status, SPEC_DEV_BAD_LENGTH);
    }
    __syncthreads();
    const unsigned long long best = fin[0], second = fin[1];
    int32_t len = 0, jb = 0;
    if (best != 0ull) {
      jb = (int32_t)(best & 0xFFFFFFFFull);
      len = min(p.L, T - 1 - jb);
    }
    // x[t] for a proposal token: one CTA holds every position it can name in
    // shared memory (window up to w1, suffix from s0); a cluster reads memory
    auto tok_at = [&](int32_t t) -> int32_t {
      if (!CLUSTER) return t < w1 ? win[t - w0] : suf[t - s0];
      return x[t];
    };
    for (int i = tid; i < p.L; i += blockDim.x)
      p.g[(int64_t)r * p.L + i] = i < len ? tok_at(jb + 1 + i) : -1;
    int32_t n_out = 0, a_out = 0, m_out = 0;
    if (best != 0ull) {
      const int32_t lb = (int32_t)(best >> 32);
      n_out = min(lb, p.n_max);
      m_out = lb;
      a_out = 1;
      if (second != 0ull) {
        const int32_t j2 = (int32_t)(second & 0xFFFFFFFFull);
        a_out = (tok_at(j2 + 1) == tok_at(jb + 1)) ? 1 : 0;
      }
    }
    if (tid == 0) {
      p.g_len[r] = len;
      p.match_n[r] = n_out;
      p.agree[r] = a_out;
      p.copy_len[r] = m_out;
    }
    if (PRICE) {
      // price this request from on-chip values (warp 0), then arrive; the CTA
      // of the last request to arrive allocates the budget for the whole batch
      __shared__ int32_t s_last;
      __shared__ int32_t s_cnt[SPEC_PACKED_ARRIVAL];  // every request's valid slots (packed arrival)
      if (tid < 32) {
        uint32_t st = 0;
        if (tid < p.L) s_ps.g[tid] = tid < len ? tok_at(jb + 1 + tid) : -1;
        const float* stab = nullptr;  // the staged table, once its copy has landed
        if (tab_smem) {
          if (mbar_wait_bounded(&tbar, 0, 1u << 22)) {
            stab = reinterpret_cast<const float*>(smem_tok + p.tab_off);
          } else {  // record it, wait (bounded) for the copy to finish, price from global memory
            st |= SPEC_DEV_TIMEOUT;
            mbar_wait_bounded(&tbar, 0, 1u << 22);
          }
        }
        __syncwarp();
        const int32_t clen = price_request_warp(p.cx, r, tid, s_ps, len, n_out, a_out, m_out, s_dl, st, stab);
        if (st) set_status(p.status, st);
        // the request's valid slots: the keys written nonzero
        const int32_t nv = __popc(__ballot_sync(0xFFFFFFFFu, tid < p.cx.L && tid < clen && tid < p.cx.mvl));
        if (tid == 0) {
          if (p.batch <= SPEC_PACKED_ARRIVAL) {
            const unsigned long long mine = (unsigned long long)(nv + 1) << (SPEC_PACKED_BITS * r);
            const unsigned long long now = atomic_add_acq_rel_u64(p.arrive64, mine) + mine;
            int last = 1;
            for (int q = 0; q < p.batch; ++q) {
              const int32_t f = (int32_t)((now >> (SPEC_PACKED_BITS * q)) & ((1u << SPEC_PACKED_BITS) - 1u));
              last &= f != 0;
              s_cnt[q] = f - 1;
            }
            s_last = last;
            if (last) *p.arrive64 = 0ull;  // ready for the next call
          } else {
            const uint32_t old = atomic_add_acq_rel(p.arrive, 1u);
            s_last = (old + 1u == (uint32_t)p.batch) ? 1 : 0;
            if (s_last) *p.arrive = 0u;  // ready for the next call
          }
        }
      }
      __syncthreads();
      if (s_last)
        select_budget_cta(p.sc, smem_tok + p.win_cap + p.suf_cap,
                          p.batch <= SPEC_PACKED_ARRIVAL ? s_cnt : nullptr);
    }
  }
  if (CLUSTER) cluster.sync();  // peers keep their shared memory until rank 0 has read it
}

}  // namespace spec

// ---------------------------------------------------------------------------
// host launcher (called from api.cu)
// ---------------------------------------------------------------------------
namespace {

template <bool PRICE>
cudaError_t launch_ngram_kernel(const spec::NgramParams& p, int64_t C, size_t smem, int32_t batch,
                                cudaStream_t stream) {
  if (C == 1) {
    // one CTA per request: a plain launch, no cluster barrier or DSMEM.  The
    // largest shared-memory carve-out, the one the verification kernel that
    // follows needs, so that the SMs keep one L1 / shared-memory split
    cudaError_t e = cudaFuncSetAttribute(spec::ngram_kernel<false, PRICE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(spec::ngram_kernel<false, PRICE>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    spec::ngram_kernel<false, PRICE><<<batch, SPEC_CTA_THREADS, smem, stream>>>(p);
    return cudaGetLastError();
  }
  cudaError_t e = cudaFuncSetAttribute(spec::ngram_kernel<true, PRICE>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(spec::ngram_kernel<true, PRICE>, cudaFuncAttributePreferredSharedMemoryCarveout,
                           (int)cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(batch * C), 1, 1);
  cfg.blockDim = dim3(SPEC_CTA_THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, spec::ngram_kernel<true, PRICE>, p);
}

// cluster size, staged-window sizes and shared memory of one launch; false if
// the history rows are too long for shared memory
bool ngram_geometry(int64_t stride, int32_t cap, int32_t extra_ints, int64_t* C_out, spec::NgramParams* p,
                    size_t* smem_out) {
  // one CTA per 8192 candidate positions (32 per thread), at most 8 (the
  // portable cluster limit); a cluster of one needs no merge traffic
  int64_t C = (stride + 8191) / 8192;
  if (C < 1) C = 1;
  if (C > 8) C = 8;
  const int64_t per = (stride + C - 1) / C;
  const int64_t win_cap = ((per + cap + 8) + 3) & ~int64_t(3);
  const int64_t suf_cap = ((int64_t)cap + 8 + 3) & ~int64_t(3);
  const size_t smem = (size_t)(win_cap + suf_cap + extra_ints) * sizeof(int32_t);
  if (smem > 200 * 1024) return false;
  p->win_cap = (int32_t)win_cap;
  p->suf_cap = (int32_t)suf_cap;
  *C_out = C;
  *smem_out = smem;
  return true;
}

void ngram_common(spec::NgramParams* p, const int32_t* hist, int64_t stride, const int32_t* hist_len,
                  int32_t batch, int32_t n_min, int32_t n_max, int32_t L, int32_t cap, int32_t* g,
                  int32_t* g_len, int32_t* match_n, int32_t* agree, int32_t* copy_len, uint32_t* status) {
  *p = spec::NgramParams{};
  p->hist = hist;
  p->stride = stride;
  p->hist_len = hist_len;
  p->batch = batch;
  p->n_min = n_min;
  p->n_max = n_max;
  p->L = L;
  p->cap = cap;
  p->g = g;
  p->g_len = g_len;
  p->match_n = match_n;
  p->agree = agree;
  p->copy_len = copy_len;
  p->status = status;
  p->use_bulk = ((reinterpret_cast<uintptr_t>(hist) & 15u) == 0 && (stride & 3) == 0) ? 1 : 0;
}

}  // namespace

extern "C" cudaError_t spec_launch_ngram(const int32_t* hist, int64_t stride, const int32_t* hist_len,
                                         int32_t batch, int32_t n_min, int32_t n_max, int32_t L,
                                         int32_t cap, int32_t* g, int32_t* g_len, int32_t* match_n,
                                         int32_t* agree, int32_t* copy_len, uint32_t* status,
                                         int num_sms, cudaStream_t stream, int* unsupported) {
  (void)num_sms;
  *unsupported = 0;
  if (batch == 0) return cudaSuccess;
  spec::NgramParams p;
  ngram_common(&p, hist, stride, hist_len, batch, n_min, n_max, L, cap, g, g_len, match_n, agree, copy_len,
               status);
  int64_t C;
  size_t smem;
  if (!ngram_geometry(stride, cap, 0, &C, &p, &smem)) {
    *unsupported = 1;
    return cudaSuccess;
  }
  return launch_ngram_kernel<false>(p, C, smem, batch, stream);
}

extern "C" cudaError_t spec_launch_draft_price(
    const int32_t* hist, int64_t stride, const int32_t* hist_len, int32_t batch, int32_t n_min, int32_t n_max,
    int32_t cap, int32_t* g, int32_t* g_len, int32_t* match_n, int32_t* agree, int32_t* copy_len, int32_t K,
    int32_t L, const int32_t* d, const float* c, const int32_t* d_len, const spec_estimator* est,
    const float* table, float lambda, int32_t budget, int32_t mvl, int32_t policy, int32_t draft_greedy,
    int32_t* chain, float* S, int32_t* chain_len, int32_t* source, int32_t* verify_len, int32_t* row_off,
    uint8_t* point_mass, uint32_t* status, uint32_t* keys, cudaStream_t stream, int* unsupported) {
  *unsupported = 0;
  spec::NgramParams p;
  ngram_common(&p, hist, stride, hist_len, batch, n_min, n_max, L, cap, g, g_len, match_n, agree, copy_len,
               status);
  p.d = d;
  p.c = c;
  p.d_len = d_len;
  p.cx.K = K;
  p.cx.L = L;
  p.cx.table = table;
  p.cx.tab_const = est->use_constant_h;
  p.cx.n_full = est->n_full;
  p.cx.m_cap = est->m_cap;
  p.cx.lambda = lambda;
  p.cx.policy = policy;
  p.cx.draft_greedy = draft_greedy;
  p.cx.chain = chain;
  p.cx.S = S;
  p.cx.chain_len = chain_len;
  p.cx.source = source;
  p.cx.point_mass = point_mass;
  p.cx.mvl = mvl;
  p.cx.keys = keys;
  p.sc.batch = batch;
  p.sc.L = L;
  p.sc.budget = budget;
  p.sc.keys = keys;
  p.sc.verify_len = verify_len;
  p.sc.row_off = row_off;
  p.arrive = status + 2;  // the third word of the workspace header
  p.arrive64 = reinterpret_cast<unsigned long long*>(status + 4);  // header words 4 and 5
  int64_t C;
  size_t smem;
  if (!ngram_geometry(stride < 1 ? 1 : stride, cap, spec::select_scratch_ints(batch, L), &C, &p, &smem)) {
    *unsupported = 1;
    return cudaSuccess;
  }
  // the Eq. (1) table into the pricing CTA's shared memory when it is whole
  // 16-byte pieces, 16-byte aligned and at most SPEC_TAB_SMEM_MAX bytes
  p.tab_off = -1;
  p.tab_bytes = 0;
  if (!est->use_constant_h) {
    const size_t tb = sizeof(float) * (size_t)L * (SPEC_TAB_N * 2 + 2 * ((size_t)est->m_cap + 1));
    const size_t off = (smem + 15) & ~(size_t)15;
    if (tb % 16 == 0 && tb <= SPEC_TAB_SMEM_MAX && (reinterpret_cast<uintptr_t>(table) & 15u) == 0 &&
        off + tb <= 200 * 1024) {
      p.tab_off = (int32_t)(off / sizeof(int32_t));
      p.tab_bytes = (uint32_t)tb;
      smem = off + tb;
    }
  }
  return launch_ngram_kernel<true>(p, C, smem, batch, stream);
}
