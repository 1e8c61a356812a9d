// common.cuh -- device helpers shared by the kernels of the round.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "spec.h"

#define SPEC_WARPS_PER_CTA 8
#define SPEC_CTA_THREADS (32 * SPEC_WARPS_PER_CTA)
#define SPEC_UNIT 2048  // vocabulary entries per work unit (one warp)

// float2 entries between two rows of the workspace's chunk partials: one per
// chunk of the finest chunking (2048 fp32 entries), then a spare entry (the
// logit at the row's draft token), rounded up to an even count so that every
// row starts on a 16-byte boundary
static inline __host__ __device__ int spec_partial_stride(int units) { return (units + 2) & ~1; }

namespace spec {

__device__ __forceinline__ void set_status(uint32_t* status, uint32_t bits) {
  if (bits) atomicOr(status, bits);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): ten rounds of two 32x32
// multiplies with the published multipliers; the key advances by the published
// Weyl increments between rounds.
__device__ __forceinline__ void philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                              uint32_t k0, uint32_t k1, uint32_t out[4]) {
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint32_t lo0 = 0xD2511F53u * c0, hi0 = __umulhi(0xD2511F53u, c0);
    const uint32_t lo1 = 0xCD9E8D57u * c2, hi1 = __umulhi(0xCD9E8D57u, c2);
    const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
    c0 = n0;
    c1 = lo1;
    c2 = n2;
    c3 = lo0;
  }
  out[0] = c0;
  out[1] = c1;
  out[2] = c2;
  out[3] = c3;
}

// uniforms of request r, position i: counter (r, i, lo32(step), hi32(step)),
// key (lo32(seed), hi32(seed)); (w >> 8) * 2^-24 is exact in fp32.
__device__ __forceinline__ void round_uniforms(uint64_t seed, uint64_t step, uint32_t r, uint32_t i,
                                               float* u, float* u2) {
  uint32_t o[4];
  philox4x32_10(r, i, (uint32_t)step, (uint32_t)(step >> 32), (uint32_t)seed,
                (uint32_t)(seed >> 32), o);
  *u = (float)(o[0] >> 8) * (1.0f / 16777216.0f);
  *u2 = (float)(o[1] >> 8) * (1.0f / 16777216.0f);
}

// float -> uint32 whose unsigned order is the float order (NaN excluded by callers)
__device__ __forceinline__ uint32_t ordered_bits(float v) {
  const uint32_t b = __float_as_uint(v);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float from_ordered_bits(uint32_t o) {
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
}
// packed argmax key: larger value first, then lower index
__device__ __forceinline__ unsigned long long argmax_key(float v, int32_t idx) {
  return ((unsigned long long)ordered_bits(v) << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)idx);
}
__device__ __forceinline__ int32_t argmax_key_index(unsigned long long k) {
  return (int32_t)(0xFFFFFFFFu - (uint32_t)(k & 0xFFFFFFFFull));
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}
__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}
// inclusive prefix sums over lanes in lane order
__device__ __forceinline__ float warp_incl_scan(float v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float t = __shfl_up_sync(0xFFFFFFFFu, v, o);
    if (lane >= o) v += t;
  }
  return v;
}
__device__ __forceinline__ double warp_incl_scan_d(double v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double t = __shfl_up_sync(0xFFFFFFFFu, v, o);
    if (lane >= o) v += t;
  }
  return v;
}

// 2^x on the SFU (MUFU.EX2); the argument is always <= 0 here
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 16-byte streaming load that does not allocate in L1
__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}


// ------------------------------------------------------------------ mbarrier + bulk copy
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
// bounded wait on phase `parity`; false when the bound ran out
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
// one-dimensional bulk async copy global -> shared, completed on `bar`
// (both addresses 16-byte aligned, bytes a multiple of 16)
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// device-scope fetch-add with acquire-release ordering (publishes this thread's
// earlier writes and, for the last arriver, makes every earlier arriver's visible)
__device__ __forceinline__ uint32_t atomic_add_acq_rel(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.add.acq_rel.gpu.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// order this thread's earlier generic-proxy accesses (and the acquire that
// preceded them) before its later bulk copies, which read through the async proxy
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async;" ::: "memory"); }

// workspace view used by device code
struct WsView {
  uint32_t* status;
  uint32_t* counter;
  uint32_t* counter2;
  uint32_t* counter3;  // per draft-row arrival counters (probabilistic drafting)
  unsigned char* record;
  unsigned long long* rowkey;
  float2* partial;   // per chunk (max, sum) of each row, spec_partial_stride(units) entries per row
  float* partial2;   // per chunk residual mass of each request's rejected position
  int32_t units;     // ceil(vocab / 2048)
  int32_t max_rows;
  int32_t max_batch;
  int32_t K;
};

}  // namespace spec
