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
// GB300 layout: one CTA of 256 threads.  The survivals of the verifiable
// slots are gathered into shared memory (no sort), then Dinkelbach's
// iteration below finds the maximising ratio with one block-wide count and
// exact fixed-point sum per round (fp64 work runs on a narrow pipe on this
// part, so only the ratio is formed in fp64).  The sums differ from a
// left-to-right fp64 sum in the last bits, so near-ties of G may resolve
// differently.
#include "common.cuh"

namespace spec {

struct BudgetParams {
  int32_t batch, L, mvl;
  const float* S;
  const int32_t* chain_len;
  double C0, p;
  int32_t* out_budget;
  float* out_lambda;
};

#define BU_THREADS 256

// A survival in [0, 1] as a multiple of 2^-48, truncated: integer sums of
// these are exact, and at most 1024 x 31 of them stay below 2^63.  The
// truncation moves a sum by less than 2^-48 per term, far less than the
// rounding of a left-to-right fp64 sum of the same terms.
__device__ __forceinline__ uint64_t fixed48(float v) {
  const uint32_t bits = __float_as_uint(v);
  const int32_t e = (int32_t)(bits >> 23);
  if (e == 0) return 0ull;  // zero or subnormal: below 2^-126
  const uint64_t m = (uint64_t)((bits & 0x7FFFFFu) | 0x800000u);
  const int32_t sh = e - 102;  // v = m 2^(e - 150), so v 2^48 = m 2^(e - 102)
  return sh >= 0 ? (m << sh) : (sh > -64 ? (m >> -sh) : 0ull);
}

__global__ void __launch_bounds__(BU_THREADS) size_budget_kernel(BudgetParams p, uint32_t* status) {
  extern __shared__ __align__(16) float s_val[];  // [batch x L]: the verifiable survivals
  __shared__ int32_t s_n;
  __shared__ unsigned long long s_part[BU_THREADS / 32];
  __shared__ int32_t s_cnt[BU_THREADS / 32];
  __shared__ float s_thr;
  __shared__ int32_t s_b, s_done;
  __shared__ double s_lam;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    s_n = 0;
    s_b = 0;
    s_lam = (double)p.batch / p.C0;  // G(0)
    s_thr = __double2float_rd(s_lam * p.p);
    s_done = 0;
  }
  __syncthreads();
  // gather the verifiable survivals (their order does not matter): batches of
  // 8 slots per thread with every load issued before any is used; one shared
  // atomic per warp and batch places them
  const int32_t nslots = p.batch * p.L;
  bool bad = false;
  for (int32_t q0 = 0; q0 < nslots; q0 += 8 * BU_THREADS) {
    float v[8];
    int32_t len[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int32_t q = q0 + j * BU_THREADS + tid;
      v[j] = q < nslots ? __ldg(p.S + q) : 0.0f;
      len[j] = q < nslots ? __ldg(p.chain_len + q / p.L) : 0;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int32_t q = q0 + j * BU_THREADS + tid;
      const int32_t k = q - (q / p.L) * p.L;
      const bool valid = q < nslots && k < min(len[j], p.mvl);
      if (valid && !(v[j] >= 0.0f && v[j] <= 1.0f)) {  // survivals are probabilities
        bad = true;
        v[j] = v[j] > 1.0f ? 1.0f : 0.0f;
      }
      const unsigned b = __ballot_sync(0xFFFFFFFFu, valid);
      int32_t base = 0;
      if (lane == 0 && b != 0u) base = atomicAdd(&s_n, __popc(b));
      base = __shfl_sync(0xFFFFFFFFu, base, 0);
      if (valid) s_val[base + __popc(b & ((1u << lane) - 1u))] = v[j];
    }
  }
  if (bad) set_status(status, SPEC_DEV_BAD_VALUE);
  __syncthreads();
  const int32_t n = s_n;
  // Dinkelbach's iteration for the ratio G = A / C: given the ratio lam of
  // the current set, the set maximising A(b) - lam C(b) takes every slot whose
  // survival exceeds lam p (a slot equal to it adds nothing, and leaving it
  // out keeps the smallest b); its ratio is the next lam.  lam rises to
  // max_b G(b) and the set stops changing there, in a few rounds.  Each round
  // is one block-wide count and exact integer sum; only the ratio itself is
  // formed in fp64, by one thread.
  for (int it = 0; it < 64 && !s_done; ++it) {
    // v > lam p for an fp32 v exactly when v > (lam p rounded down to fp32)
    const float thr = s_thr;
    int32_t cnt = 0;
    uint64_t sum = 0;
    for (int32_t i = tid; i < n; i += BU_THREADS) {
      const float v = s_val[i];
      if (v > thr) {
        ++cnt;
        sum += fixed48(v);
      }
    }
    cnt = __reduce_add_sync(0xFFFFFFFFu, cnt);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
    if (lane == 0) {
      s_part[warp] = sum;
      s_cnt[warp] = cnt;
    }
    __syncthreads();
    if (tid == 0) {
      int32_t c = 0;
      uint64_t sm = 0;
#pragma unroll
      for (int w = 0; w < BU_THREADS / 32; ++w) {
        c += s_cnt[w];
        sm += s_part[w];
      }
      const double lam_new = ((double)p.batch + (double)sm * 0x1p-48) / (p.C0 + p.p * (double)c);
      if (c == s_b || !(lam_new > s_lam)) {
        s_done = 1;  // the set stopped changing (or the ratio stopped rising)
      } else {
        s_b = c;
        s_lam = lam_new;
        s_thr = __double2float_rd(lam_new * p.p);
      }
    }
    __syncthreads();
  }
  if (tid == 0) {
    *p.out_budget = s_b;
    *p.out_lambda = (float)(s_lam * p.p);
  }
}

// The same sizing with every slot in registers when the batch has at most
// BU_REG_SLOTS slots: thread t holds slots t + 256 j (j < 8), each survival
// with its fixed-point value (-1 marks a slot that may not be verified), all
// loaded at once (no compaction), so a round is eight register terms per
// thread, one warp reduction and thread 0's ratio between two barriers.
#define BU_REG_SLOTS 2048
__global__ void __launch_bounds__(BU_THREADS) size_budget_reg_kernel(BudgetParams p, uint32_t* status) {
  constexpr int J = BU_REG_SLOTS / BU_THREADS;
  __shared__ unsigned long long s_part[BU_THREADS / 32];
  __shared__ int32_t s_cnt[BU_THREADS / 32];
  __shared__ float s_thr;
  __shared__ int32_t s_done;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int32_t nslots = p.batch * p.L;
  float v[J];
  uint64_t f[J];
  bool bad = false;
  {
    // slot q = tid + 256 j: request q / L and position q % L, advanced without division
    int32_t rr[J], kk[J];
    int32_t r = tid / p.L, k = tid - r * p.L;
    const int32_t dr = BU_THREADS / p.L, dk = BU_THREADS - dr * p.L;
#pragma unroll
    for (int j = 0; j < J; ++j) {
      rr[j] = r;
      kk[j] = k;
      k += dk;
      r += dr;
      if (k >= p.L) {
        k -= p.L;
        ++r;
      }
    }
    int32_t len[J];
#pragma unroll
    for (int j = 0; j < J; ++j) {  // every load issued before any is used
      const int32_t q = tid + BU_THREADS * j;
      len[j] = q < nslots ? __ldg(p.chain_len + rr[j]) : 0;
      v[j] = q < nslots ? __ldg(p.S + q) : -1.0f;
    }
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const int32_t q = tid + BU_THREADS * j;
      float x = v[j];
      if (q < nslots && kk[j] < min(len[j], p.mvl)) {
        if (!(x >= 0.0f && x <= 1.0f)) {  // survivals are probabilities
          bad = true;
          x = x > 1.0f ? 1.0f : 0.0f;
        }
      } else {
        x = -1.0f;
      }
      v[j] = x;
      f[j] = x >= 0.0f ? fixed48(x) : 0ull;
    }
  }
  if (__any_sync(0xFFFFFFFFu, bad) && lane == 0) set_status(status, SPEC_DEV_BAD_VALUE);
  // Dinkelbach's iteration, as in size_budget_kernel
  double lam = (double)p.batch / p.C0;  // G(0) (thread 0's copy is the one used)
  int32_t b = 0;
  if (tid == 0) {
    s_thr = __double2float_rd(lam * p.p);
    s_done = 0;
  }
  __syncthreads();
  for (int it = 0; it < 64; ++it) {
    const float thr = s_thr;
    int32_t cnt = 0;
    uint64_t sum = 0;
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const bool in = v[j] > thr;  // slots that may not be verified hold -1
      cnt += in ? 1 : 0;
      sum += in ? f[j] : 0ull;
    }
    cnt = __reduce_add_sync(0xFFFFFFFFu, cnt);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
    if (lane == 0) {
      s_part[warp] = sum;
      s_cnt[warp] = cnt;
    }
    __syncthreads();
    if (tid == 0) {
      int32_t c = 0;
      uint64_t sm = 0;
#pragma unroll
      for (int w = 0; w < BU_THREADS / 32; ++w) {
        c += s_cnt[w];
        sm += s_part[w];
      }
      const double lam_new = ((double)p.batch + (double)sm * 0x1p-48) / (p.C0 + p.p * (double)c);
      if (c == b || !(lam_new > lam)) {
        s_done = 1;  // the set stopped changing (or the ratio stopped rising)
      } else {
        b = c;
        lam = lam_new;
        s_thr = __double2float_rd(lam_new * p.p);
      }
    }
    __syncthreads();
    if (s_done) break;
  }
  if (tid == 0) {
    *p.out_budget = b;
    *p.out_lambda = (float)(lam * p.p);
  }
}

}  // namespace spec

extern "C" size_t spec_budget_smem_bytes(int32_t batch, int32_t L) {
  const int64_t n = (int64_t)batch * L;
  return (size_t)(n < 1 ? 1 : n) * sizeof(float);
}

extern "C" cudaError_t spec_launch_size_budget(int32_t batch, int32_t L, const float* S, const int32_t* chain_len,
                                               int32_t mvl, double C0, double p, int32_t* out_budget,
                                               float* out_lambda, uint32_t* status, cudaStream_t stream) {
  spec::BudgetParams bp;
  bp.batch = batch;
  bp.L = L;
  bp.mvl = mvl;
  const size_t smem = spec_budget_smem_bytes(batch, L);
  bp.S = S;
  bp.chain_len = chain_len;
  bp.C0 = C0;
  bp.p = p;
  bp.out_budget = out_budget;
  bp.out_lambda = out_lambda;
  if ((int64_t)batch * L <= BU_REG_SLOTS) {  // every slot in registers
    spec::size_budget_reg_kernel<<<1, BU_THREADS, 0, stream>>>(bp, status);
    return cudaGetLastError();
  }
  cudaError_t e = cudaFuncSetAttribute(spec::size_budget_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  spec::size_budget_kernel<<<1, BU_THREADS, smem, stream>>>(bp, status);
  return cudaGetLastError();
}
