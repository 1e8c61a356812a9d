// ngram.cu -- step 1 of the round: n-gram prompt lookup.
//
// Hybrid Spark sec. 4.1 ("One step"): the n-gram drafter proposes up to L
// tokens following the longest earlier occurrence of the request's last
// n_min..n_max tokens (sec. 5.1: longest match wins); sec. 4.2 defines the
// features n (match length), a (runner-up agreement) and m (copy length,
// capped).  Every earlier end position j <= T-2 has a match length l(j), the
// common-suffix length of x[..j] and x[..T-1] capped at copy_cap; candidates
// (l(j) >= n_min) rank by (l(j), j) descending.
//
// GB300 layout: one thread-block cluster per request.  The cluster's CTAs
// split the candidate positions into contiguous chunks; each CTA stages its
// chunk (plus a copy_cap halo behind it) and the request's last copy_cap
// tokens into shared memory with one-dimensional bulk async copies completed
// on an mbarrier, compares suffixes from shared memory (one position per
// thread, early exit on the first mismatch), and reduces a top-2 of packed
// (l, j) keys with warp shuffles.  Cluster rank 0 merges the CTAs' top-2
// through distributed shared memory and writes the proposal and features.
#include <cooperative_groups.h>

#include "common.cuh"

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
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// bounded wait on phase `parity` of an mbarrier; false when the bound ran out
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint32_t max_iter) {
  const uint32_t addr = smem_u32(bar);
  for (uint32_t it = 0; it < max_iter; ++it) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(addr), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

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

__global__ void __launch_bounds__(SPEC_CTA_THREADS) ngram_kernel(NgramParams p) {
  extern __shared__ __align__(16) int32_t smem_tok[];
  __shared__ __align__(8) uint64_t bar;
  __shared__ unsigned long long warp_best[SPEC_WARPS_PER_CTA][2];
  __shared__ unsigned long long cta_best[2];
  __shared__ int32_t s_flag;

  cg::cluster_group cluster = cg::this_cluster();
  const int C = (int)cluster.num_blocks();
  const int rank = (int)cluster.block_rank();
  const int r = blockIdx.x / C;
  const int tid = threadIdx.x;
  const int32_t* x = p.hist + (int64_t)r * p.stride;

  const int32_t T = p.hist_len[r];
  const bool valid = (T >= 0) && ((int64_t)T <= p.stride);
  const int32_t nc = valid && T >= 2 ? T - 1 : 0;  // candidate end positions 0..T-2
  const int32_t per = (nc + C - 1) / C;
  const int32_t j0 = min(nc, rank * per);
  const int32_t j1 = min(nc, j0 + per);
  const bool work = j0 < j1;

  // staged ranges, rounded to 4-token (16-byte) boundaries
  const int32_t w0 = max(0, j0 - p.cap + 1) & ~3;
  const int32_t w1 = (j1 + 3) & ~3;
  const int32_t s0 = max(0, T - p.cap) & ~3;
  const int32_t s1 = (T + 3) & ~3;
  int32_t* win = smem_tok;               // x[w0 .. w1)
  int32_t* suf = smem_tok + p.win_cap;   // x[s0 .. s1)

  if (tid == 0) s_flag = 0;
  if (work) {
    if (p.use_bulk) {
      if (tid == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(smem_u32(&bar)) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
      }
      __syncthreads();
      if (tid == 0) {
        const uint32_t wb = (uint32_t)(w1 - w0) * 4u, sb = (uint32_t)(s1 - s0) * 4u;
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(&bar)),
                     "r"(wb + sb)
                     : "memory");
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

  unsigned long long b1 = 0ull, b2 = 0ull;  // packed (l << 32 | j); 0 = none
  if (work && s_flag == 0) {
    const int32_t* wv = win - w0;  // wv[t] = x[t]
    const int32_t* sv = suf - s0;
    const int32_t last = sv[T - 1];
    for (int32_t j = j0 + tid; j < j1; j += blockDim.x) {
      if (wv[j] != last) continue;
      const int32_t lim = min(p.cap, j + 1);
      int32_t l = 1;
      while (l < lim && wv[j - l] == sv[T - 1 - l]) ++l;
      if (l >= p.n_min) top2_insert(b1, b2, ((unsigned long long)l << 32) | (uint32_t)j);
    }
  }
  warp_top2(b1, b2);
  const int warp = tid >> 5, lane = tid & 31;
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
  cluster.sync();

  if (rank == 0) {
    __shared__ unsigned long long fin[2];
    if (tid == 0) {
      unsigned long long c1 = 0ull, c2 = 0ull;
      for (int q = 0; q < C; ++q) {
        const unsigned long long* peer = cluster.map_shared_rank(cta_best, q);
        top2_insert(c1, c2, peer[0]);
        top2_insert(c1, c2, peer[1]);
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
    for (int i = tid; i < p.L; i += blockDim.x)
      p.g[(int64_t)r * p.L + i] = i < len ? x[jb + 1 + i] : -1;
    if (tid == 0) {
      if (best == 0ull) {
        p.g_len[r] = 0;
        p.match_n[r] = 0;
        p.agree[r] = 0;
        p.copy_len[r] = 0;
      } else {
        const int32_t lb = (int32_t)(best >> 32);
        p.g_len[r] = len;
        p.match_n[r] = min(lb, p.n_max);
        p.copy_len[r] = lb;
        int32_t a = 1;
        if (second != 0ull) {
          const int32_t j2 = (int32_t)(second & 0xFFFFFFFFull);
          a = (x[j2 + 1] == x[jb + 1]) ? 1 : 0;
        }
        p.agree[r] = a;
      }
    }
  }
  cluster.sync();  // peers keep their shared memory until rank 0 has read it
}

}  // namespace spec

// ---------------------------------------------------------------------------
// host launcher (called from api.cu)
// ---------------------------------------------------------------------------
extern "C" cudaError_t spec_launch_ngram(const int32_t* hist, int64_t stride, const int32_t* hist_len,
                                         int32_t batch, int32_t n_min, int32_t n_max, int32_t L,
                                         int32_t cap, int32_t* g, int32_t* g_len, int32_t* match_n,
                                         int32_t* agree, int32_t* copy_len, uint32_t* status,
                                         int num_sms, cudaStream_t stream, int* unsupported) {
  *unsupported = 0;
  if (batch == 0) return cudaSuccess;
  // cluster size: enough CTAs to cover the GPU, at least 256 positions each,
  // at most 8 (the portable cluster limit)
  int64_t c_len = (stride + 4095) / 4096;
  int64_t c_occ = (2 * (int64_t)num_sms + batch - 1) / batch;
  int64_t C = c_len > c_occ ? c_len : c_occ;
  if (C > stride / 256) C = stride / 256;
  if (C < 1) C = 1;
  if (C > 8) C = 8;
  const int64_t per = (stride + C - 1) / C;
  const int64_t win_cap = ((per + cap + 8) + 3) & ~int64_t(3);
  const int64_t suf_cap = ((int64_t)cap + 8 + 3) & ~int64_t(3);
  const size_t smem = (size_t)(win_cap + suf_cap) * sizeof(int32_t);
  if (smem > 200 * 1024) {
    *unsupported = 1;
    return cudaSuccess;
  }
  spec::NgramParams p;
  p.hist = hist;
  p.stride = stride;
  p.hist_len = hist_len;
  p.batch = batch;
  p.n_min = n_min;
  p.n_max = n_max;
  p.L = L;
  p.cap = cap;
  p.g = g;
  p.g_len = g_len;
  p.match_n = match_n;
  p.agree = agree;
  p.copy_len = copy_len;
  p.status = status;
  p.win_cap = (int32_t)win_cap;
  p.suf_cap = (int32_t)suf_cap;
  p.use_bulk = ((reinterpret_cast<uintptr_t>(hist) & 15u) == 0 && (stride & 3) == 0) ? 1 : 0;

  cudaError_t e = cudaFuncSetAttribute(spec::ngram_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
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
  return cudaLaunchKernelEx(&cfg, spec::ngram_kernel, p);
}
