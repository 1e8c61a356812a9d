// budget.cu -- sizing the next verification budget from one step's survivals.
//
// Hybrid Spark sec. 2 (adaptive verification), sec. 4.3 Eq. (2), sec. 4.4 and
// App. F: over the slots that may be verified (k < min(chain_len, max_verify_len))
// with survivals s_(1) >= s_(2) >= ...,
//   G(b) = (batch + sum_{i <= b} s_(i)) / (C0 + p b),  b* = the smallest
//   maximiser over b in [0, #slots],  lambda = G(b*) p.
// The host passes b* and lambda to the pricing step two steps later (App. O);
// this kernel produces them on the device so that the host only copies two
// scalars back, asynchronously.
//
// GB300 layout: one CTA of 1024 threads.  The survivals of the verifiable
// slots are gathered into shared memory, sorted descending by a bitonic sort
// over the next power of two, then each thread takes a contiguous segment of
// the sorted list: segment sums in fp64, one block scan, a walk that forms
// A(b) and G(b) for its b, and a block-wide argmax (largest G, then smallest
// b).  The sums associate by segment, not left to right, so G may differ from
// a sequential sum in the last bits.
#include "common.cuh"

namespace spec {

#define BU_THREADS 1024
#define BU_WARPS (BU_THREADS / 32)

struct BudgetParams {
  int32_t batch, L, mvl, n_pad;
  const float* S;
  const int32_t* chain_len;
  double C0, p;
  int32_t* out_budget;
  float* out_lambda;
};

__global__ void __launch_bounds__(BU_THREADS, 1) size_budget_kernel(BudgetParams p) {
  extern __shared__ __align__(16) float s_val[];  // [n_pad]
  __shared__ int32_t s_n;
  __shared__ double s_part[BU_WARPS];
  __shared__ double s_bestG[BU_WARPS];
  __shared__ int32_t s_bestb[BU_WARPS];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) s_n = 0;
  for (int32_t i = tid; i < p.n_pad; i += BU_THREADS) s_val[i] = -1.0f;  // below every survival
  __syncthreads();
  // gather the verifiable survivals (their order does not matter: they are sorted next)
  const int32_t nslots = p.batch * p.L;
  for (int32_t q = tid; q < nslots; q += BU_THREADS) {
    const int32_t r = q / p.L, k = q - r * p.L;
    int32_t len = __ldg(p.chain_len + r);
    len = len < p.mvl ? len : p.mvl;
    if (k < len) s_val[atomicAdd(&s_n, 1)] = __ldg(p.S + q);
  }
  __syncthreads();
  const int32_t n = s_n;
  // bitonic sort, descending
  for (int32_t size = 2; size <= p.n_pad; size <<= 1) {
    for (int32_t stride = size >> 1; stride > 0; stride >>= 1) {
      for (int32_t i = tid; i < p.n_pad / 2; i += BU_THREADS) {
        const int32_t lo = 2 * i - (i & (stride - 1));  // pairs (lo, lo + stride)
        const int32_t hi = lo + stride;
        const bool desc = ((lo & size) == 0);
        const float a = s_val[lo], b = s_val[hi];
        if (desc ? (a < b) : (a > b)) {
          s_val[lo] = b;
          s_val[hi] = a;
        }
      }
      __syncthreads();
    }
  }
  // contiguous segments of the sorted list: sums, scan, then G(b) for b in the segment
  const int32_t per = (n + BU_THREADS - 1) / BU_THREADS;
  const int32_t b0 = tid * per, b1 = min(n, b0 + per);
  double seg = 0.0;
  for (int32_t i = b0; i < b1; ++i) seg += (double)s_val[i];
  double incl = seg;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) s_part[warp] = incl;
  __syncthreads();
  double before = 0.0;
  for (int w = 0; w < warp; ++w) before += s_part[w];
  double A = (double)p.batch + (before + (incl - seg));  // A at b = b0
  double bestG = -1.0;
  int32_t bestb = 0;
  if (tid == 0) {
    bestG = A / p.C0;  // b = 0
    bestb = 0;
  }
  for (int32_t i = b0; i < b1; ++i) {
    A += (double)s_val[i];
    const int32_t b = i + 1;
    const double G = A / (p.C0 + p.p * (double)b);
    if (G > bestG) {
      bestG = G;
      bestb = b;
    }
  }
  // argmax over the block: largest G, ties to the smallest b
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const double g2 = __shfl_down_sync(0xFFFFFFFFu, bestG, o);
    const int32_t b2 = __shfl_down_sync(0xFFFFFFFFu, bestb, o);
    if (g2 > bestG || (g2 == bestG && b2 < bestb)) {
      bestG = g2;
      bestb = b2;
    }
  }
  if (lane == 0) {
    s_bestG[warp] = bestG;
    s_bestb[warp] = bestb;
  }
  __syncthreads();
  if (tid == 0) {
    double g = s_bestG[0];
    int32_t b = s_bestb[0];
    for (int w = 1; w < BU_WARPS; ++w)
      if (s_bestG[w] > g || (s_bestG[w] == g && s_bestb[w] < b)) {
        g = s_bestG[w];
        b = s_bestb[w];
      }
    *p.out_budget = b;
    *p.out_lambda = (float)(g * p.p);
  }
}

}  // namespace spec

extern "C" size_t spec_budget_smem_bytes(int32_t batch, int32_t L) {
  int64_t n = 1;
  while (n < (int64_t)batch * L) n <<= 1;
  return (size_t)(n < 2 ? 2 : n) * sizeof(float);
}

extern "C" cudaError_t spec_launch_size_budget(int32_t batch, int32_t L, const float* S, const int32_t* chain_len,
                                               int32_t mvl, double C0, double p, int32_t* out_budget,
                                               float* out_lambda, cudaStream_t stream) {
  spec::BudgetParams bp;
  bp.batch = batch;
  bp.L = L;
  bp.mvl = mvl;
  const size_t smem = spec_budget_smem_bytes(batch, L);
  bp.n_pad = (int32_t)(smem / sizeof(float));
  bp.S = S;
  bp.chain_len = chain_len;
  bp.C0 = C0;
  bp.p = p;
  bp.out_budget = out_budget;
  bp.out_lambda = out_lambda;
  cudaError_t e = cudaFuncSetAttribute(spec::size_budget_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  spec::size_budget_kernel<<<1, BU_THREADS, smem, stream>>>(bp);
  return cudaGetLastError();
}
