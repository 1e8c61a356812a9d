// verify.cu -- steps 3 and 4 of the round: chain verification and greedy tree
// verification over full-vocabulary logit rows.
//
// Chain (Hybrid Spark sec. 2, App. H; the fixed-cost parallel drafter page's
// verification rule): accept y_i iff u_i < min(1, p_i(y_i)/q_i(y_i)), q a
// point mass for greedy / n-gram drafts; at the first rejection draw from
// norm(max(0, p_i - q_i)); after all acceptances draw a bonus from p_{ell+1};
// T = 0 accepts iff y_i = argmax.  r accepted => r + 1 tokens.
// Tree (AdaSpark sec. 2.2): a node is accepted iff its token equals the argmax
// at its parent's row and its parent is accepted; commit the path and the
// argmax after it.
//
// GB300 layout.  The HBM-bound part is one pass over every verify row.  One
// CTA per SM, 12 warps each; the work is the sequence of 8 KB chunks of the
// rows (4096 bf16 / 2048 fp32 entries) in (request, row, chunk) order, and
// every warp takes an equal contiguous range of it.  Each warp streams its
// range through its own 8 KB shared-memory stage filled by one-dimensional
// bulk async copies (completion on an mbarrier, bounded wait): it moves a
// landed chunk into registers and refills the stage at once, so its next
// copy is in flight while it computes.  One 8 KB copy per warp (96 KB per
// SM, 15 MB over the GPU) keeps HBM busy; deeper rings measured slower, as
// longer memory queues widen the spread of the warps' finish times.  Per
// chunk a warp
// produces
//   greedy rows:  a packed 64-bit (ordered value, ~index) key; keys of one
//                 row fold in registers and reach the row's workspace key with
//                 one atomicMax per run of the row (largest value, lowest
//                 index);
//   sampled rows: (max, sum of 2^((z - max) log2e / T)) per 2048-entry unit
//                 in the workspace.
// Each request has an arrival counter; the warp that completes a request's
// last chunk (acquire-release atomic, no waiting) finalizes it: argmax
// compare or Philox accept tests, and for a draw the inverse CDF in
// vocabulary order located first over the units' sums and then inside the
// one unit that holds the crossing (a second read of 4-8 KB, not of the row).
// A draw from max(0, p - q) needs both normalisers first; those requests are
// finished by a second, small kernel over the rejected (p, q) row pairs.
#include <cuda_bf16.h>

#include "common.cuh"

namespace spec {

enum { MODE_CHAIN_GREEDY = 0, MODE_CHAIN_SAMPLE = 1, MODE_TREE = 2 };

// streaming kernel: 12 warps per CTA, one CTA per SM, each warp with its own
// 8 KB stage (96 KB of shared memory in flight per SM)
#define VR_WARPS 12
#define VR_THREADS (32 * VR_WARPS)
enum { KIND_POINT = 0, KIND_BONUS = 1, KIND_Q = 2 };

struct VerifyParams {
  int32_t batch, vocab;
  const void* logits;      // target logits (chain) or tree logits
  const int32_t* row_off;  // chain: row_off [batch+1]; tree: node_off [batch+1]
  int32_t max_rows;
  const void* draft;  // [batch x K x vocab] or null
  int32_t K;
  const int32_t* chain;
  int32_t L;
  const int32_t* verify_len;
  const uint8_t* pm;
  int32_t use_q;  // draft logits present and T > 0
  float c;        // log2(e) / T
  uint64_t seed, step;
  int32_t* out_tokens;
  int32_t* n_accepted;
  int32_t* n_emitted;
  float* dbg_ratio;
  float* dbg_u;
  float* dbg_resid;
  const int32_t* tok;
  const int32_t* parent;
  int32_t max_nodes;
  int32_t* path;
  int32_t* accept_len;
  int32_t units;   // ceil(vocab / SPEC_UNIT)
  int32_t vec_ok;  // every row starts on a 16-byte boundary
  WsView ws;
};

// resample record of one request (64 bytes), written by the finalizer of a
// request whose draw needs max(0, p - q)
struct __align__(16) Record {
  int32_t flag, pos, prow, qrow;
  float mp, sp, mq, sq;
  float u2;
  int32_t pad[7];
};

// ------------------------------------------------------------------ loading
// strided layout: lane-interleaved 16-byte vectors (coalesced); element j of
// a lane sits at unit offset idx_strided<DT>(lane, j)
template <int DT>
__device__ __forceinline__ int idx_strided(int lane, int j, bool vec) {
  if (!vec) return lane + 32 * j;
  if (DT == 1) return 8 * (lane + 32 * (j >> 3)) + (j & 7);
  return 4 * (lane + 32 * (j >> 2)) + (j & 3);
}

// 64 values of one unit, fp32, missing entries = -inf
template <int DT>
__device__ __forceinline__ void load_unit(const void* row, int e0, int n_el, bool vec, int lane,
                                          float v[64]) {
  if (vec) {
    if (DT == 1) {
      const uint16_t* rp = static_cast<const uint16_t*>(row) + e0;
      uint4 w[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int vv = lane + 32 * k;
        if (8 * vv < n_el)
          w[k] = ldg_stream(rp + 8 * vv);
        else
          w[k] = make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        v[8 * k + 0] = bf16_lo(w[k].x);
        v[8 * k + 1] = bf16_hi(w[k].x);
        v[8 * k + 2] = bf16_lo(w[k].y);
        v[8 * k + 3] = bf16_hi(w[k].y);
        v[8 * k + 4] = bf16_lo(w[k].z);
        v[8 * k + 5] = bf16_hi(w[k].z);
        v[8 * k + 6] = bf16_lo(w[k].w);
        v[8 * k + 7] = bf16_hi(w[k].w);
      }
    } else {
      const float* rp = static_cast<const float*>(row) + e0;
      uint4 w[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const int vv = lane + 32 * k;
        if (4 * vv < n_el)
          w[k] = ldg_stream(rp + 4 * vv);
        else
          w[k] = make_uint4(0xFF800000u, 0xFF800000u, 0xFF800000u, 0xFF800000u);
      }
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        v[4 * k + 0] = __uint_as_float(w[k].x);
        v[4 * k + 1] = __uint_as_float(w[k].y);
        v[4 * k + 2] = __uint_as_float(w[k].z);
        v[4 * k + 3] = __uint_as_float(w[k].w);
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < 64; ++j) {
      const int i = lane + 32 * j;
      float x = -INFINITY;
      if (i < n_el) {
        if (DT == 1)
          x = __uint_as_float((uint32_t)__ldg(static_cast<const uint16_t*>(row) + e0 + i) << 16);
        else
          x = __ldg(static_cast<const float*>(row) + e0 + i);
      }
      v[j] = x;
    }
  }
}

// contiguous layout for the sampling rescan: lane l holds unit offsets
// [64 l, 64 l + 64) in order; missing entries = -inf
template <int DT>
__device__ __forceinline__ void load_unit_contig(const void* row, int e0, int n_el, bool vec,
                                                 int lane, float v[64]) {
  const int b = 64 * lane;
  if (vec && b + 64 <= n_el) {
    if (DT == 1) {
      const uint4* rp = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(row) + e0 + b);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint4 w = __ldcg(rp + k);
        v[8 * k + 0] = bf16_lo(w.x);
        v[8 * k + 1] = bf16_hi(w.x);
        v[8 * k + 2] = bf16_lo(w.y);
        v[8 * k + 3] = bf16_hi(w.y);
        v[8 * k + 4] = bf16_lo(w.z);
        v[8 * k + 5] = bf16_hi(w.z);
        v[8 * k + 6] = bf16_lo(w.w);
        v[8 * k + 7] = bf16_hi(w.w);
      }
    } else {
      const uint4* rp = reinterpret_cast<const uint4*>(static_cast<const float*>(row) + e0 + b);
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const uint4 w = __ldcg(rp + k);
        v[4 * k + 0] = __uint_as_float(w.x);
        v[4 * k + 1] = __uint_as_float(w.y);
        v[4 * k + 2] = __uint_as_float(w.z);
        v[4 * k + 3] = __uint_as_float(w.w);
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < 64; ++j) {
      const int i = b + j;
      float x = -INFINITY;
      if (i < n_el) {
        if (DT == 1)
          x = __uint_as_float((uint32_t)__ldcg(static_cast<const unsigned short*>(row) + e0 + i) << 16);
        else
          x = __ldcg(static_cast<const float*>(row) + e0 + i);
      }
      v[j] = x;
    }
  }
}

template <int DT>
__device__ __forceinline__ float load_one(const void* row, int64_t i) {
  if (DT == 1) return __uint_as_float((uint32_t)__ldcg(static_cast<const unsigned short*>(row) + i) << 16);
  return __ldcg(static_cast<const float*>(row) + i);
}

// ------------------------------------------------------------------ per unit
// A chunk is 8 KB of one row (4096 bf16 / 2048 fp32 entries).  Each lane holds
// NV 16-byte vectors of it: vector vv = lane + 32 k covers chunk offsets
// [8 vv, 8 vv + 8) (bf16) or [4 vv, 4 vv + 4) (fp32); vectors past the row's
// end hold -inf.
template <int DT>
struct Vec {
  static constexpr int NV = 16;                // vectors per lane per chunk
  static constexpr int PER = DT == 1 ? 8 : 4;  // entries per vector
  static constexpr int CH = 32 * NV * PER;     // entries per chunk: 4096 bf16 / 2048 fp32
  static constexpr int BYTES = 8192;           // bytes per chunk (one pipeline stage)
  static constexpr int STAGES = 1;  // copies in flight per warp
  static constexpr int SUB = CH / SPEC_UNIT;   // 2048-entry units per chunk
  static constexpr uint32_t NEG = DT == 1 ? 0xFF80FF80u : 0xFF800000u;
};

template <int DT>
__device__ __forceinline__ void vec_load_global(const void* unit, int n_el, int lane, uint4 (&w)[Vec<DT>::NV]) {
#pragma unroll
  for (int k = 0; k < Vec<DT>::NV; ++k) {
    const int vv = lane + 32 * k;
    w[k] = (Vec<DT>::PER * vv < n_el) ? ldg_stream(static_cast<const uint4*>(unit) + vv)
                                      : make_uint4(Vec<DT>::NEG, Vec<DT>::NEG, Vec<DT>::NEG, Vec<DT>::NEG);
  }
}

template <int DT>
__device__ __forceinline__ void vec_load_smem(const void* unit, int n_el, int lane, uint4 (&w)[Vec<DT>::NV]) {
  if (n_el == Vec<DT>::CH) {  // no bounds tests on a full chunk
#pragma unroll
    for (int k = 0; k < Vec<DT>::NV; ++k) w[k] = static_cast<const uint4*>(unit)[lane + 32 * k];
    return;
  }
#pragma unroll
  for (int k = 0; k < Vec<DT>::NV; ++k) {
    const int vv = lane + 32 * k;
    w[k] = (Vec<DT>::PER * vv < n_el) ? static_cast<const uint4*>(unit)[vv]
                                      : make_uint4(Vec<DT>::NEG, Vec<DT>::NEG, Vec<DT>::NEG, Vec<DT>::NEG);
  }
}

__device__ __forceinline__ float vec_elem_f32(const uint4& v, int e) {
  const uint32_t x = e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w;
  return __uint_as_float(x);
}

// argmax of one unit: packed key of (max, lowest unit offset) or 0 when the unit
// holds only NaN; `bad` collects NaN / +Inf (warp-uniform after the call).
// Per-vector maxima first (independent, so the dependency chains stay short),
// NaN-propagating so that one test per lane finds a NaN; the NaN-ignoring
// maximum is recomputed only for a unit that holds one.
__device__ __forceinline__ __nv_bfloat162 as_bf2(uint32_t x) { return *reinterpret_cast<__nv_bfloat162*>(&x); }
__device__ __forceinline__ uint32_t bf2_bits(__nv_bfloat162 x) { return *reinterpret_cast<uint32_t*>(&x); }

template <int DT>
__device__ __forceinline__ unsigned long long unit_argmax_vec(const uint4 (&w)[Vec<DT>::NV], int n_el, int lane,
                                                              int& bad) {
  constexpr int NV = Vec<DT>::NV;
  float vmax[NV];  // max of each vector (NaN-propagating)
  if (DT == 1) {
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const __nv_bfloat162 a = __hmax2_nan(as_bf2(w[k].x), as_bf2(w[k].y));
      const __nv_bfloat162 b = __hmax2_nan(as_bf2(w[k].z), as_bf2(w[k].w));
      const __nv_bfloat162 c = __hmax2_nan(a, b);
      vmax[k] = fmaxf(__low2float(c), __high2float(c));
      if (__low2float(c) != __low2float(c) || __high2float(c) != __high2float(c)) vmax[k] = __int_as_float(0x7FC00000);
    }
  } else {
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const float a = __uint_as_float(w[k].x), b = __uint_as_float(w[k].y);
      const float c = __uint_as_float(w[k].z), d = __uint_as_float(w[k].w);
      const float m = fmaxf(fmaxf(a, b), fmaxf(c, d));
      vmax[k] = ((a != a) | (b != b) | (c != c) | (d != d)) ? __int_as_float(0x7FC00000) : m;
    }
  }
  // NaN-propagating tree over the vectors
  float t[NV];
#pragma unroll
  for (int k = 0; k < NV; ++k) t[k] = vmax[k];
#pragma unroll
  for (int h = NV / 2; h > 0; h >>= 1)
#pragma unroll
    for (int k = 0; k < h; ++k) t[k] = (t[k] != t[k] || t[k + h] != t[k + h]) ? __int_as_float(0x7FC00000)
                                                                              : fmaxf(t[k], t[k + h]);
  float lane_max = t[0];
  const bool has_nan = lane_max != lane_max;
  if (__any_sync(0xFFFFFFFFu, has_nan)) {
    // rare: a unit with NaN.  Per-vector NaN-ignoring maxima.
    bad = 1;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      float m = -INFINITY;
      if (DT == 1) {
        const uint32_t ws[4] = {w[k].x, w[k].y, w[k].z, w[k].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) m = fmaxf(m, fmaxf(bf16_lo(ws[q]), bf16_hi(ws[q])));
      } else {
        m = fmaxf(fmaxf(__uint_as_float(w[k].x), __uint_as_float(w[k].y)),
                  fmaxf(__uint_as_float(w[k].z), __uint_as_float(w[k].w)));
      }
      vmax[k] = m;
    }
    lane_max = -INFINITY;
#pragma unroll
    for (int k = 0; k < NV; ++k) lane_max = fmaxf(lane_max, vmax[k]);
  }
  const float wm = warp_max(lane_max);
  int idx = 0x7FFFFFFF;
  if (lane_max == wm) {
    // the first vector whose maximum is wm, then the first entry in it
    int kf = -1;
#pragma unroll
    for (int k = NV - 1; k >= 0; --k)
      if (vmax[k] == wm && Vec<DT>::PER * (lane + 32 * k) < n_el) kf = k;
    if (kf >= 0) {
      uint4 v = w[0];
#pragma unroll
      for (int k = 1; k < NV; ++k)
        if (k == kf) v = w[k];
      const int base = Vec<DT>::PER * (lane + 32 * kf);
      if (DT == 1) {
        const uint32_t ws[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 3; q >= 0; --q) {
          if (bf16_hi(ws[q]) == wm) idx = base + 2 * q + 1;
          if (bf16_lo(ws[q]) == wm) idx = base + 2 * q;
        }
      } else {
#pragma unroll
        for (int e = 3; e >= 0; --e)
          if (vec_elem_f32(v, e) == wm) idx = base + e;
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) idx = min(idx, __shfl_xor_sync(0xFFFFFFFFu, idx, o));
  bad |= __any_sync(0xFFFFFFFFu, wm == INFINITY);
  return idx == 0x7FFFFFFF ? 0ull : argmax_key(wm, idx);
}

// the k-th vector of a register-held chunk, by a jump table rather than a chain
// of selects (only the lane holding the maximum takes this path)
template <int NV>
__device__ __forceinline__ uint4 pick_vec(const uint4 (&w)[NV], int k) {
  uint4 v = w[0];
  switch (k) {
#define SPEC_PICK(i) \
  case i:            \
    if (i < NV) v = w[i < NV ? i : 0]; \
    break;
    SPEC_PICK(0) SPEC_PICK(1) SPEC_PICK(2) SPEC_PICK(3) SPEC_PICK(4) SPEC_PICK(5) SPEC_PICK(6) SPEC_PICK(7)
    SPEC_PICK(8) SPEC_PICK(9) SPEC_PICK(10) SPEC_PICK(11) SPEC_PICK(12) SPEC_PICK(13) SPEC_PICK(14) SPEC_PICK(15)
#undef SPEC_PICK
    default:
      break;
  }
  return v;
}

// bf16 argmax of one register-held chunk.  Packed bf16x2 maxima, NaN-propagating
// so that one test per lane finds a NaN; the lane holding the maximum locates
// its vector from the per-vector maxima and then the entry inside it.
__device__ __forceinline__ unsigned long long chunk_argmax_bf16(const uint4 (&w)[Vec<1>::NV], int n_el, int lane,
                                                                int& bad) {
  constexpr int NV = Vec<1>::NV;
  __nv_bfloat162 vm[NV];
#pragma unroll
  for (int k = 0; k < NV; ++k)
    vm[k] = __hmax2_nan(__hmax2_nan(as_bf2(w[k].x), as_bf2(w[k].y)), __hmax2_nan(as_bf2(w[k].z), as_bf2(w[k].w)));
  __nv_bfloat162 t[NV];
#pragma unroll
  for (int k = 0; k < NV; ++k) t[k] = vm[k];
#pragma unroll
  for (int h = NV / 2; h > 0; h >>= 1)
#pragma unroll
    for (int k = 0; k < h; ++k) t[k] = __hmax2_nan(t[k], t[k + h]);
  const float lo = __low2float(t[0]), hi = __high2float(t[0]);
  float lane_max = fmaxf(lo, hi);
  if (__any_sync(0xFFFFFFFFu, (lo != lo) || (hi != hi))) {
    // rare: the chunk holds a NaN.  NaN-ignoring per-vector maxima instead.
    bad = 1;
#pragma unroll
    for (int k = 0; k < NV; ++k)
      vm[k] = __hmax2(__hmax2(as_bf2(w[k].x), as_bf2(w[k].y)), __hmax2(as_bf2(w[k].z), as_bf2(w[k].w)));
    lane_max = -INFINITY;
#pragma unroll
    for (int k = 0; k < NV; ++k) lane_max = fmaxf(lane_max, fmaxf(__low2float(vm[k]), __high2float(vm[k])));
  }
  const float wm = warp_max(lane_max);
  int idx = 0x7FFFFFFF;
  if (lane_max == wm) {
    const __nv_bfloat162 wm2 = __float2bfloat162_rn(wm);  // exact: wm is a bf16 value
    int kf = -1;
#pragma unroll
    for (int k = NV - 1; k >= 0; --k)
      if (__heq2_mask(vm[k], wm2) != 0u && 8 * (lane + 32 * k) < n_el) kf = k;
    if (kf >= 0) {
      const uint4 x = pick_vec<NV>(w, kf);
      const int base = 8 * (lane + 32 * kf);
      const uint32_t ws[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int q = 3; q >= 0; --q) {
        if (bf16_hi(ws[q]) == wm) idx = base + 2 * q + 1;
        if (bf16_lo(ws[q]) == wm) idx = base + 2 * q;
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) idx = min(idx, __shfl_xor_sync(0xFFFFFFFFu, idx, o));
  bad |= __any_sync(0xFFFFFFFFu, wm == INFINITY);
  return idx == 0x7FFFFFFF ? 0ull : argmax_key(wm, idx);
}

// (max, sum 2^((z - max) c)) of one unit; an all -inf unit gives (-inf, 0).
// Several independent partial maxima and sums keep the dependency chains short.
template <int DT, int KB, int KN>
__device__ __forceinline__ float2 unit_softmax_vec(const uint4 (&w)[Vec<DT>::NV], float c, int& bad) {
  float vm[KN];
#pragma unroll
  for (int k = 0; k < KN; ++k) {
    const uint4& x = w[KB + k];
    if (DT == 1) {
      const __nv_bfloat162 a = __hmax2(as_bf2(x.x), as_bf2(x.y));
      const __nv_bfloat162 b = __hmax2(as_bf2(x.z), as_bf2(x.w));
      const __nv_bfloat162 m2 = __hmax2(a, b);
      vm[k] = fmaxf(__low2float(m2), __high2float(m2));
    } else {
      vm[k] = fmaxf(fmaxf(__uint_as_float(x.x), __uint_as_float(x.y)),
                    fmaxf(__uint_as_float(x.z), __uint_as_float(x.w)));
    }
  }
#pragma unroll
  for (int h = KN / 2; h > 0; h >>= 1)
#pragma unroll
    for (int k = 0; k < h; ++k) vm[k] = fmaxf(vm[k], vm[k + h]);
  const float m = warp_max(vm[0]);
  float s = 0.0f;
  if (m != -INFINITY) {
    const float mc = m * c;
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int k = 0; k < KN; ++k) {
      const uint4& x = w[KB + k];
      const uint32_t ws[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (DT == 1) {
          acc[q] += ex2(fmaf(bf16_lo(ws[q]), c, -mc)) + ex2(fmaf(bf16_hi(ws[q]), c, -mc));
        } else {
          acc[q] += ex2(fmaf(__uint_as_float(ws[q]), c, -mc));
        }
      }
    }
    s = (acc[0] + acc[1]) + (acc[2] + acc[3]);
  }
  s = warp_sum(s);
  bad |= (!(s == s) || m == INFINITY) ? 1 : 0;
  return make_float2(m, s);
}

// the same two reductions for rows that are not 16-byte aligned (scalar loads,
// element j of a lane at unit offset lane + 32 j)
template <int DT>
__device__ __forceinline__ unsigned long long unit_argmax_scalar(const void* unit, int n_el, int lane, int& bad) {
  float v[64];
  load_unit<DT>(unit, 0, n_el, false, lane, v);
  float lm = -INFINITY;
  int nan = 0;
#pragma unroll
  for (int j = 0; j < 64; ++j) {
    lm = fmaxf(lm, v[j]);
    nan |= (v[j] != v[j]);
  }
  const float wm = warp_max(lm);
  int idx = 0x7FFFFFFF;
  if (lm == wm) {
#pragma unroll
    for (int j = 0; j < 64; ++j) {
      const int i = lane + 32 * j;
      if (i < n_el && v[j] == wm && i < idx) idx = i;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) idx = min(idx, __shfl_xor_sync(0xFFFFFFFFu, idx, o));
  bad |= __any_sync(0xFFFFFFFFu, nan || wm == INFINITY);
  return idx == 0x7FFFFFFF ? 0ull : argmax_key(wm, idx);
}

template <int DT>
__device__ __forceinline__ float2 unit_softmax_scalar(const void* unit, int n_el, int lane, float c, int& bad) {
  float v[64];
  load_unit<DT>(unit, 0, n_el, false, lane, v);
  float lm = -INFINITY;
#pragma unroll
  for (int j = 0; j < 64; ++j) lm = fmaxf(lm, v[j]);
  const float m = warp_max(lm);
  float s = 0.0f;
  if (m != -INFINITY) {
    const float mc = m * c;
#pragma unroll
    for (int j = 0; j < 64; ++j) s += ex2(fmaf(v[j], c, -mc));
  }
  s = warp_sum(s);
  bad |= (!(s == s) || m == INFINITY) ? 1 : 0;
  return make_float2(m, s);
}

// ------------------------------------------------------------------ helpers
// (m, s) pairs merged: s rescaled to the larger max (empty pairs have m = -inf)
__device__ __forceinline__ void merge_ms(float& m, float& s, float m2, float s2, float c) {
  const float nm = fmaxf(m, m2);
  if (nm == -INFINITY) return;
  s = (m == -INFINITY ? 0.0f : s * ex2((m - nm) * c)) + (m2 == -INFINITY ? 0.0f : s2 * ex2((m2 - nm) * c));
  m = nm;
}

// (max, sum) of R rows from their unit partials, by the whole warp at once.
// Row k (its partials at slot_of(k); none when negative) is merged by G lanes,
// G the largest power of two with R G <= 32: each lane takes every G-th unit
// in batches of MB independent loads (one memory round trip per batch, with an
// online rescale), then the G lanes combine by shuffles.  More than 32 rows
// take several rounds.  Lane l receives row want_a(l)'s result in *a and row
// want_b(l)'s in *b (negative: none, (-inf, 0)).
template <typename SlotFn>
__device__ __forceinline__ void merge_rows_warp(const VerifyParams& p, int R, SlotFn slot_of, int lane, int want_a,
                                                float2* a, int want_b, float2* b) {
  constexpr int MB = 20;
  int G = 1;
  while (G < 32 && R * 2 * G <= 32) G <<= 1;
  const int rpr = 32 / G, sub = lane & (G - 1);
  *a = make_float2(-INFINITY, 0.0f);
  *b = make_float2(-INFINITY, 0.0f);
  for (int k0 = 0; k0 < R; k0 += rpr) {
    const int k = k0 + lane / G;
    const int slot = k < R ? slot_of(k) : -1;
    float m = -INFINITY, s = 0.0f;
    if (slot >= 0) {
      const float2* pr = &p.ws.partial[(int64_t)slot * p.ws.units];
      for (int u0 = sub; u0 < p.units; u0 += MB * G) {
        float2 t[MB];
#pragma unroll
        for (int q = 0; q < MB; ++q) {
          const int u = u0 + q * G;
          t[q] = u < p.units ? __ldcg(&pr[u]) : make_float2(-INFINITY, 0.0f);
        }
        float bm = -INFINITY;
#pragma unroll
        for (int q = 0; q < MB; ++q) bm = fmaxf(bm, t[q].x);
        if (bm == -INFINITY) continue;
        const float nm = fmaxf(m, bm);
        float acc = (m == -INFINITY) ? 0.0f : s * ex2((m - nm) * p.c);
#pragma unroll
        for (int q = 0; q < MB; ++q)
          if (t[q].x != -INFINITY) acc += t[q].y * ex2((t[q].x - nm) * p.c);
        m = nm;
        s = acc;
      }
    }
    for (int o = G >> 1; o >= 1; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xFFFFFFFFu, m, o), s2 = __shfl_xor_sync(0xFFFFFFFFu, s, o);
      merge_ms(m, s, m2, s2, p.c);
    }
    // rows k0 .. k0 + rpr - 1 sit at lanes (k - k0) G
    const bool in_a = want_a >= k0 && want_a < k0 + rpr, in_b = want_b >= k0 && want_b < k0 + rpr;
    const float ma = __shfl_sync(0xFFFFFFFFu, m, in_a ? (want_a - k0) * G : 0);
    const float sa = __shfl_sync(0xFFFFFFFFu, s, in_a ? (want_a - k0) * G : 0);
    const float mb = __shfl_sync(0xFFFFFFFFu, m, in_b ? (want_b - k0) * G : 0);
    const float sb = __shfl_sync(0xFFFFFFFFu, s, in_b ? (want_b - k0) * G : 0);
    if (in_a) *a = make_float2(ma, sa);
    if (in_b) *b = make_float2(mb, sb);
  }
}

// Inverse CDF over unit weights w_u (unit order), at the fraction u of their
// total: returns the unit holding the crossing of t = u * total, the weight
// before it, the total and t.  Each lane owns `per` consecutive units, so lane
// order is unit order; a lane keeps its first four weights in registers for
// the walk that locates the crossing.  The sums run in fp32 (the weights are
// fp32 products, and fp64 work runs on a narrow pipe on this part).
struct Crossing {
  int unit;
  float before;  // weight of the units before `unit`; -1: t at or above the total
  float total;
  float t;
};

template <typename WFn>
__device__ __forceinline__ Crossing find_unit(int units, float u, int lane, WFn wfn) {
  const int per = (units + 31) / 32;
  const int u0 = lane * per;
  float w4[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) w4[q] = (q < per && u0 + q < units) ? wfn(u0 + q) : 0.0f;
  float lsum = 0.0f;
  int last_pos = -1;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    lsum += w4[q];
    if (w4[q] > 0.0f) last_pos = u0 + q;
  }
  for (int q = 4; q < per; ++q) {
    const int uu = u0 + q;
    if (uu < units) {
      const float w = wfn(uu);
      lsum += w;
      if (w > 0.0f) last_pos = uu;
    }
  }
  const float incl = warp_incl_scan(lsum);
  const float excl = incl - lsum;
  Crossing c;
  c.total = __shfl_sync(0xFFFFFFFFu, incl, 31);
  c.t = u * c.total;
  const float t = c.t;
  const unsigned hit = __ballot_sync(0xFFFFFFFFu, incl > t && lsum > 0.0f);
  if (hit) {
    const int src = __ffs(hit) - 1;
    int unit = -1;
    float before = 0.0f;
    if (lane == src) {
      float run = excl;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float w = w4[q];
        if (unit < 0 && q < per && u0 + q < units) {
          if (run + w > t && w > 0.0f) {
            unit = u0 + q;
            before = run;
          }
          run += w;
        }
      }
      for (int q = 4; q < per && unit < 0; ++q) {
        const int uu = u0 + q;
        if (uu >= units) break;
        const float w = wfn(uu);
        if (run + w > t && w > 0.0f) {
          unit = uu;
          before = run;
        }
        run += w;
      }
      if (unit < 0) {  // rounding inside the lane: its last unit with mass
        unit = last_pos;
        float wl = 0.0f;
        if (last_pos >= 0) {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            if (u0 + q == last_pos) wl = w4[q];
          if (last_pos >= u0 + 4) wl = wfn(last_pos);
        }
        before = incl - wl;
      }
    }
    c.unit = __shfl_sync(0xFFFFFFFFu, unit, src);
    c.before = __shfl_sync(0xFFFFFFFFu, before, src);
  } else {
    // t at or above the total (rounding): the last unit with mass
    const unsigned has = __ballot_sync(0xFFFFFFFFu, last_pos >= 0);
    const int src = has ? 31 - __clz(has) : 0;
    const int lp = __shfl_sync(0xFFFFFFFFu, last_pos, src);
    c.unit = lp < 0 ? 0 : lp;
    c.before = -1.0f;  // marker: take the last positive entry of the unit
  }
  return c;
}

// inside one unit: the smallest index whose running sum (from `before`)
// exceeds t, over residual values r[64] in contiguous lane layout.  Returns
// (index within the unit, r at that index); falls back to the last positive.
// The sums inside the unit run from the unit's start, against t - before.
__device__ __forceinline__ int find_in_unit(const float r[64], float before, float t, int lane, float* r_at) {
  float a0 = 0.0f, a1 = 0.0f, a2 = 0.0f, a3 = 0.0f;
#pragma unroll
  for (int j = 0; j < 64; j += 4) {
    a0 += r[j];
    a1 += r[j + 1];
    a2 += r[j + 2];
    a3 += r[j + 3];
  }
  const float lsum = (a0 + a1) + (a2 + a3);
  const float incl = warp_incl_scan(lsum);
  const float excl = incl - lsum;
  const float tr = t - before;
  int pick = -1;
  float rv = 0.0f;
  const bool last_mode = before < 0.0f;
  const unsigned hit = last_mode ? 0u : __ballot_sync(0xFFFFFFFFu, incl > tr && lsum > 0.0f);
  if (hit) {
    const int src = __ffs(hit) - 1;
    if (lane == src) {
      // unrolled without an early exit, so r[] stays in registers
      float run = excl, lastv = 0.0f;
      int lastp = -1;
#pragma unroll
      for (int j = 0; j < 64; ++j) {
        const float x = r[j];
        if (x > 0.0f) {
          lastp = j;
          lastv = x;
        }
        run += x;
        if (pick < 0 && run > tr && x > 0.0f) {
          pick = 64 * lane + j;
          rv = x;
        }
      }
      if (pick < 0 && lastp >= 0) {
        pick = 64 * lane + lastp;
        rv = lastv;
      }
    }
    pick = __shfl_sync(0xFFFFFFFFu, pick, src);
    rv = __shfl_sync(0xFFFFFFFFu, rv, src);
  } else {
    int lastp = -1;
    for (int j = 0; j < 64; ++j)
      if (r[j] > 0.0f) lastp = j;
    const unsigned has = __ballot_sync(0xFFFFFFFFu, lastp >= 0);
    if (has) {
      const int src = 31 - __clz(has);
      pick = __shfl_sync(0xFFFFFFFFu, 64 * lane + lastp, src);
      float mine = 0.0f;
#pragma unroll
      for (int j = 0; j < 64; ++j)
        if (j == lastp) mine = r[j];
      rv = __shfl_sync(0xFFFFFFFFu, mine, src);
    } else {
      pick = 0;
      rv = 0.0f;
    }
  }
  *r_at = rv;
  return pick;
}


// ---- one unit's weights for a draw, in compact code.  A draw runs once per
// request, from cold instruction caches, so these loops stay rolled: lane l
// owns the unit's entries [64 l, 64 l + 64), read through L1 in 16-byte
// vectors (one memory round trip for the first pass; the rest hit L1).  The
// weight of entry z is 2^(z c - mc), 0 for -inf and for the excluded index.
template <int DT>
__device__ __forceinline__ void unpack_vec(const uint4& w, float (&x)[DT == 1 ? 8 : 4]) {
  if (DT == 1) {
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      x[2 * q] = bf16_lo(ws[q]);
      x[2 * q + 1] = bf16_hi(ws[q]);
    }
  } else {
    x[0] = __uint_as_float(w.x);
    x[1] = __uint_as_float(w.y);
    x[2] = __uint_as_float(w.z);
    x[3] = __uint_as_float(w.w);
  }
}

template <int DT>
__device__ __forceinline__ float entry_l1(const void* row, int64_t i) {
  if (DT == 1) return __uint_as_float((uint32_t)__ldca(static_cast<const unsigned short*>(row) + i) << 16);
  return __ldca(static_cast<const float*>(row) + i);
}

// the lane's entries in order, from running sum `run`, with weight wf(k, x)
// of unit entry k with logit x: mode 0 returns their total; mode 1 stops at
// the first entry whose running sum exceeds t (its unit index in *pick,
// weight in *w_at), else gives the last entry with positive weight (-1 if none)
template <int DT, int MODE, typename WF>
__device__ __forceinline__ float unit_lane_pass(const void* row, int e0, int n_el, bool vec, int lane, float run,
                                                float t, int* pick, float* w_at, WF wf) {
  constexpr int PER = DT == 1 ? 8 : 4;
  constexpr size_t ESZ = DT == 1 ? 2 : 4;
  const int b = 64 * lane;
  const int cnt = min(64, n_el - b);
  float sum = 0.0f, lastw = 0.0f;
  int last = -1;
  if (MODE == 1) *pick = -1;
  if (cnt <= 0) return 0.0f;
  auto take = [&](int k, float w) -> bool {  // true: crossing found
    if (MODE == 0) {
      sum += w;
    } else if (w > 0.0f) {
      run += w;
      last = k;
      lastw = w;
      if (run > t) {
        *pick = k;
        *w_at = w;
        return true;
      }
    }
    return false;
  };
  if (vec && cnt == 64) {
    const uint4* rp = reinterpret_cast<const uint4*>(static_cast<const char*>(row) + (size_t)(e0 + b) * ESZ);
    if (DT != 1)  // the lane's 256 bytes span two 128-byte lines: ask for both at once
      asm volatile("prefetch.global.L1 [%0];" ::"l"(rp + 8));
#pragma unroll 2
    for (int i = 0; i < 64 / PER; ++i) {
      float x[PER];
      unpack_vec<DT>(__ldca(rp + i), x);
#pragma unroll
      for (int e = 0; e < PER; ++e) {
        const int k = b + i * PER + e;
        if (take(k, wf(k, x[e]))) return 0.0f;
      }
    }
  } else {
    for (int j = 0; j < cnt; ++j) {
      const int k = b + j;
      const float x = entry_l1<DT>(row, (int64_t)e0 + k);
      if (take(k, wf(k, x))) return 0.0f;
    }
  }
  if (MODE == 1) {
    *pick = last;
    *w_at = lastw;
  }
  return sum;
}

// inverse CDF inside one unit: the first entry (in index order) whose running
// sum from `before` exceeds t; the last entry with positive weight when
// rounding leaves none (before < 0: always the last).  Returns the unit index
// and *w_at its weight.
template <int DT, typename WF>
__device__ __forceinline__ int unit_draw(const void* row, int e0, int n_el, bool vec, int lane, float before, float t,
                                         float* w_at, WF wf) {
  int pk;
  float wa;
  const float lsum = unit_lane_pass<DT, 0>(row, e0, n_el, vec, lane, 0.0f, 0.0f, &pk, &wa, wf);
  const float incl = warp_incl_scan(lsum);
  const float tr = t - before;
  const unsigned hit = before < 0.0f ? 0u : __ballot_sync(0xFFFFFFFFu, incl > tr && lsum > 0.0f);
  const unsigned has = __ballot_sync(0xFFFFFFFFu, lsum > 0.0f);
  int src;
  float run, tt;
  if (hit) {
    src = __ffs(hit) - 1;
    run = incl - lsum;
    tt = tr;
  } else {
    src = has ? 31 - __clz(has) : 0;
    run = 0.0f;
    tt = INFINITY;  // no crossing: the lane's last positive entry
  }
  int pick = -1;
  float w = 0.0f;
  if (lane == src) unit_lane_pass<DT, 1>(row, e0, n_el, vec, lane, run, tt, &pick, &w, wf);
  pick = __shfl_sync(0xFFFFFFFFu, pick, src);
  *w_at = __shfl_sync(0xFFFFFFFFu, w, src);
  return pick < 0 ? 0 : pick;
}

// the weight 2^(z c - mc) of a logit z (0 for -inf and for entry `skip`)
struct SoftW {
  float c, mc;
  int skip;
  __device__ __forceinline__ float operator()(int k, float x) const {
    return (k == skip || x == -INFINITY) ? 0.0f : ex2(fmaf(x, c, -mc));
  }
};

// ------------------------------------------------------------------ finalize
__device__ __forceinline__ void write_invalid_chain(const VerifyParams& p, int r, int lane) {
  for (int j = lane; j <= p.L; j += 32) p.out_tokens[(int64_t)r * (p.L + 1) + j] = -1;
  for (int j = lane; j < p.L; j += 32) {
    if (p.dbg_ratio) p.dbg_ratio[(int64_t)r * p.L + j] = -1.0f;
    if (p.dbg_u) p.dbg_u[(int64_t)r * p.L + j] = -1.0f;
  }
  if (lane == 0) {
    p.n_accepted[r] = 0;
    p.n_emitted[r] = 0;
    if (p.dbg_resid) p.dbg_resid[r] = -1.0f;
  }
}

__device__ __forceinline__ int q_slot_of(const VerifyParams& p, int r, int i /*1-based*/) {
  return p.max_rows + r * p.K + (i - 1);
}

template <int DT>
__device__ void finalize_chain_greedy(const VerifyParams& p, int r, int base, int ell, int lane) {
  const int32_t* y = p.chain + (int64_t)r * p.L;
  // both loads first, then use them
  unsigned long long key = 0ull;
  if (lane <= ell) key = __ldcg(&p.ws.rowkey[base + lane]);
  const int yi = lane < ell ? __ldcg(y + lane) : -1;
  const int a = key ? argmax_key_index(key) : 0;  // an all-NaN row: 0 (flagged already)
  if (lane <= ell) p.ws.rowkey[base + lane] = 0ull;
  const bool tested = lane < ell;
  if (tested && (yi < 0 || yi >= p.vocab)) set_status(p.ws.status, SPEC_DEV_BAD_TOKEN);
  const bool ok = tested && yi == a;
  const unsigned fail = __ballot_sync(0xFFFFFFFFu, tested && !ok);
  const int stop = fail ? __ffs(fail) - 1 : ell;  // 0-based row of the emitted argmax
  const int n_acc = stop;
  const int a_stop = __shfl_sync(0xFFFFFFFFu, a, stop);
  for (int j = lane; j <= p.L; j += 32) {
    int t = -1;
    if (j < n_acc) t = j == lane ? yi : y[j];  // lane j holds y[j] (L < 32)
    if (j == n_acc) t = a_stop;
    p.out_tokens[(int64_t)r * (p.L + 1) + j] = t;
  }
  for (int j = lane; j < p.L; j += 32) {
    const bool tj = j <= stop && j < ell;
    if (p.dbg_ratio) p.dbg_ratio[(int64_t)r * p.L + j] = tj ? (j < n_acc ? 1.0f : 0.0f) : -1.0f;
    if (p.dbg_u) p.dbg_u[(int64_t)r * p.L + j] = tj ? 0.0f : -1.0f;
  }
  if (lane == 0) {
    p.n_accepted[r] = n_acc;
    p.n_emitted[r] = n_acc + 1;
    if (p.dbg_resid) p.dbg_resid[r] = 1.0f;
  }
}

template <int DT>
__device__ void finalize_chain_sample(const VerifyParams& p, int r, int base, int ell, int lane) {
  const int32_t* y = p.chain + (int64_t)r * p.L;
  const uint8_t* pmr = p.pm ? p.pm + (int64_t)r * p.L : nullptr;
  // lane i-1 tests position i: its token's logits are loaded first, so that
  // those loads overlap the merges below
  const bool tested = lane < ell;
  int use_q_lane = 0, yi = -1;
  float zp = 0.0f, zq = 0.0f;
  if (tested) {
    yi = y[lane];
    use_q_lane = (p.use_q && pmr && pmr[lane] == 0 && lane + 1 <= p.K) ? 1 : 0;
    if (yi >= 0 && yi < p.vocab) {
      zp = load_one<DT>(p.logits, (int64_t)(base + lane) * p.vocab + yi);
      if (use_q_lane) zq = load_one<DT>(p.draft, ((int64_t)r * p.K + lane) * p.vocab + yi);
    }
  }
  // (max, sum) of the p rows 0 .. ell (row k = lane k) and of the q rows of
  // the positions that carry one (row ell + 1 + j = the j-th such position),
  // merged by the whole warp at once
  const unsigned qmask = __ballot_sync(0xFFFFFFFFu, use_q_lane);
  const int R = ell + 1 + __popc(qmask);
  auto slot_of = [&](int k) -> int {
    if (k <= ell) return base + k;
    unsigned mm = qmask;
    int i = 0;
    for (int t = 0; t <= k - ell - 1; ++t) {
      i = __ffs(mm) - 1;
      mm &= mm - 1u;
    }
    return q_slot_of(p, r, i + 1);
  };
  float2 prow, qrow;
  merge_rows_warp(p, R, slot_of, lane, lane <= ell ? lane : -1, &prow,
                  use_q_lane ? ell + 1 + __popc(qmask & ((1u << lane) - 1u)) : -1, &qrow);
  const float mrow = prow.x, srow = prow.y, mq = qrow.x, sq = qrow.y;
  // accept tests
  float ratio = -1.0f, u = -1.0f, u2 = 0.0f;
  bool acc = false;
  if (tested) {
    round_uniforms(p.seed, p.step, (uint32_t)r, (uint32_t)(lane + 1), &u, &u2);
    if (yi < 0 || yi >= p.vocab) {
      set_status(p.ws.status, SPEC_DEV_BAD_TOKEN);
      ratio = 0.0f;
    } else {
      const float py = ex2((zp - mrow) * p.c) / srow;
      if (use_q_lane) {
        const float qy = ex2((zq - mq) * p.c) / sq;
        ratio = py / qy;
      } else {
        ratio = py;
      }
    }
    acc = (ratio >= 1.0f) || (u < ratio);
  }
  const unsigned fail = __ballot_sync(0xFFFFFFFFu, tested && !acc);
  const int stop = fail ? __ffs(fail) - 1 : ell;  // 0-based row that is sampled
  const int n_acc = stop;
  // dbg and accepted tokens
  for (int j = lane; j < p.L; j += 32) {
    const bool tj = j <= stop && j < ell;
    if (p.dbg_ratio) p.dbg_ratio[(int64_t)r * p.L + j] = tj ? ratio : -1.0f;
    if (p.dbg_u) p.dbg_u[(int64_t)r * p.L + j] = tj ? u : -1.0f;
  }
  for (int j = lane; j <= p.L; j += 32)
    if (j != n_acc) p.out_tokens[(int64_t)r * (p.L + 1) + j] = j < n_acc ? (j == lane ? yi : y[j]) : -1;
  if (lane == 0) {
    p.n_accepted[r] = n_acc;
    p.n_emitted[r] = n_acc + 1;
  }
  // the draw
  float u2_stop;
  {
    float ua, ub;
    round_uniforms(p.seed, p.step, (uint32_t)r, (uint32_t)(stop + 1), &ua, &ub);
    u2_stop = ub;
  }
  const float m = __shfl_sync(0xFFFFFFFFu, mrow, stop);
  const float s = __shfl_sync(0xFFFFFFFFu, srow, stop);
  const bool rejected = stop < ell;
  const int y_stop = rejected ? __shfl_sync(0xFFFFFFFFu, yi, stop) : -1;
  const int q_stop = rejected ? __shfl_sync(0xFFFFFFFFu, use_q_lane, stop) : 0;
  if (q_stop) {
    // needs both normalisers: finished by resample_kernel
    const float mqs = __shfl_sync(0xFFFFFFFFu, mq, stop);
    const float sqs = __shfl_sync(0xFFFFFFFFu, sq, stop);
    if (lane == 0) {
      Record* rec = reinterpret_cast<Record*>(p.ws.record) + r;
      Record t;
      t.flag = 1;
      t.pos = stop + 1;
      t.prow = base + stop;
      t.qrow = q_slot_of(p, r, stop + 1);
      t.mp = m;
      t.sp = s;
      t.mq = mqs;
      t.sq = sqs;
      t.u2 = u2_stop;
      *rec = t;
    }
    return;
  }
  const int slot = base + stop;
  const void* row = static_cast<const char*>(p.logits) + (int64_t)slot * p.vocab * (DT == 1 ? 2 : 4);
  const int yv = (y_stop >= 0 && y_stop < p.vocab) ? y_stop : -1;  // point mass to remove
  const int u_y = yv >= 0 ? yv / SPEC_UNIT : -1;
  const bool vec = p.vec_ok != 0;
  const float zy = __shfl_sync(0xFFFFFFFFu, zp, stop);  // y's logit, loaded for its test
  auto w_plain = [&](int uu) -> float {
    const float2 t = __ldcg(&p.ws.partial[(int64_t)slot * p.ws.units + uu]);
    if (t.x == -INFINITY) return 0.0f;
    return t.y * ex2((t.x - m) * p.c);
  };
  // The unit holding y, with y removed: first its partial less y's own term
  // (no rescan).  Where the residual mass is under 1/16 of the row's, that
  // difference can lose the precision the draw needs, and the unit is
  // rescanned instead.
  const float w_self = yv >= 0 ? ex2(fmaf(zy, p.c, -m * p.c)) : 0.0f;
  auto w_fast = [&](int uu) -> float {
    const float w = w_plain(uu);
    return uu == u_y ? fmaxf(w - w_self, 0.0f) : w;
  };
  Crossing cr = find_unit(p.units, u2_stop, lane, w_fast);
  const float mc = m * p.c;
  if (yv >= 0 && !(cr.total >= 0.0625f * s)) {
    const int ey = u_y * SPEC_UNIT;
    int pk;
    float wa;
    const float w_y = warp_sum(unit_lane_pass<DT, 0>(row, ey, min(SPEC_UNIT, p.vocab - ey), vec, lane, 0.0f, 0.0f,
                                                     &pk, &wa, SoftW{p.c, mc, yv - ey}));
    cr = find_unit(p.units, u2_stop, lane, [&](int uu) -> float { return uu == u_y ? w_y : w_plain(uu); });
  }
  // the draw removes y when the residual mass (unnormalised) exceeds 1e-30
  // of the row's mass, else it falls back to p itself
  const bool remove = yv >= 0 && cr.total > 1e-30f * s;
  if (yv >= 0 && !remove) cr = find_unit(p.units, u2_stop, lane, w_plain);
  const int e0 = cr.unit * SPEC_UNIT;
  float r_at;
  const int pick = unit_draw<DT>(row, e0, min(SPEC_UNIT, p.vocab - e0), vec, lane, cr.before, cr.t, &r_at,
                                 SoftW{p.c, mc, remove ? yv - e0 : -1});
  if (lane == 0) {
    p.out_tokens[(int64_t)r * (p.L + 1) + n_acc] = e0 + pick;
    if (p.dbg_resid) p.dbg_resid[r] = r_at / cr.total;
  }
}

__device__ void finalize_tree(const VerifyParams& p, int r, int base, int n, int lane) {
  // node data in registers: lane holds nodes lane + 32 q
  int a[SPEC_MAX_TREE_NODES / 32], par[SPEC_MAX_TREE_NODES / 32], tk[SPEC_MAX_TREE_NODES / 32];
  bool bad_tree = false, bad_tok = false;
#pragma unroll
  for (int q = 0; q < SPEC_MAX_TREE_NODES / 32; ++q) {
    const int j = lane + 32 * q;
    a[q] = 0;
    par[q] = -2;
    tk[q] = -1;
    if (j < n) {
      unsigned long long* kp = &p.ws.rowkey[base + j];
      const unsigned long long key = __ldcg(kp);
      a[q] = key ? argmax_key_index(key) : 0;
      *kp = 0ull;
      par[q] = p.parent[base + j];
      tk[q] = p.tok[base + j];
      if (j == 0 ? par[q] != -1 : (par[q] < 0 || par[q] >= j)) bad_tree = true;
      if (j > 0 && (tk[q] < 0 || tk[q] >= p.vocab)) bad_tok = true;
    }
  }
  const bool any_bad = __any_sync(0xFFFFFFFFu, bad_tree);
  if (__any_sync(0xFFFFFFFFu, bad_tok) && lane == 0) set_status(p.ws.status, SPEC_DEV_BAD_TOKEN);
  int32_t* path = p.path + (int64_t)r * p.max_nodes;
  int32_t* out = p.out_tokens + (int64_t)r * p.max_nodes;
  if (any_bad) {
    for (int j = lane; j < p.max_nodes; j += 32) {
      path[j] = -1;
      out[j] = -1;
    }
    if (lane == 0) {
      set_status(p.ws.status, SPEC_DEV_BAD_TREE);
      p.accept_len[r] = -1;
    }
    return;
  }
  auto get = [&](const int* arr, int j) -> int {
    int v = 0;
#pragma unroll
    for (int q = 0; q < SPEC_MAX_TREE_NODES / 32; ++q) {
      const int t = __shfl_sync(0xFFFFFFFFu, arr[q], j & 31);
      if (q == (j >> 5)) v = t;
    }
    return v;
  };
  int cur = 0, len = 1;
  if (lane == 0) path[0] = 0;
  int acur = get(a, 0);
  for (;;) {
    int next = -1;
#pragma unroll
    for (int q = 0; q < SPEC_MAX_TREE_NODES / 32; ++q) {
      const int j = lane + 32 * q;
      const unsigned m = __ballot_sync(0xFFFFFFFFu, j > cur && j < n && par[q] == cur && tk[q] == acur);
      if (m && next < 0) next = 32 * q + __ffs(m) - 1;
    }
    if (next < 0) break;
    const int tn = get(tk, next);
    if (lane == 0) {
      out[len - 1] = tn;
      path[len] = next;
    }
    ++len;
    cur = next;
    acur = get(a, cur);
  }
  if (lane == 0) {
    out[len - 1] = acur;
    p.accept_len[r] = len - 1;
  }
  for (int j = len + lane; j < p.max_nodes; j += 32) path[j] = -1;
  for (int j = len + lane; j < p.max_nodes; j += 32) out[j] = -1;
}

// ------------------------------------------------------------------ main kernel
// A cursor walks work rows in increasing order and locates each row's data.
struct Cursor {
  int r, item, slot;
  const char* row;
};

template <int MODE>
__device__ __forceinline__ void locate(const VerifyParams& p, const int32_t* s_pre, const int32_t* s_base,
                                       const int32_t* s_len, int item, size_t esz, Cursor& c) {
  if (item == c.item) return;
  while (s_pre[c.r + 1] <= item) ++c.r;
  c.item = item;
  const int li = item - s_pre[c.r];
  const int len = s_len[c.r];
  if (MODE == MODE_TREE || li <= len) {
    c.slot = s_base[c.r] + li;
    c.row = static_cast<const char*>(p.logits) + (int64_t)c.slot * p.vocab * esz;
  } else {
    // the (li - len)-th position (1-based) that carries a draft distribution
    int want = li - len, pos = 1;
    const uint8_t* pmr = p.pm + (int64_t)c.r * p.L;
    for (int i = 1; i <= len && i <= p.K; ++i)
      if (pmr[i - 1] == 0 && --want == 0) {
        pos = i;
        break;
      }
    c.slot = q_slot_of(p, c.r, pos);
    c.row = static_cast<const char*>(p.draft) + ((int64_t)c.r * p.K + pos - 1) * p.vocab * esz;
  }
}

template <int DT, int MODE>
__global__ void __launch_bounds__(VR_THREADS, 1) verify_rows_kernel(VerifyParams p) {
  constexpr int ST = Vec<DT>::STAGES, UB = Vec<DT>::BYTES;
  constexpr size_t esz = DT == 1 ? 2 : 4;
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  unsigned char* stage = smem + (size_t)warp * ST * UB;  // this warp's ring of unit buffers
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)VR_WARPS * ST * UB) + warp * ST;
  int32_t* s_pre = reinterpret_cast<int32_t*>(smem + (size_t)VR_WARPS * ST * (UB + 8));
  int32_t* s_base = s_pre + p.batch + 1;
  int32_t* s_len = s_base + p.batch;
  __shared__ int32_t s_part[VR_WARPS];

  const int B = p.batch;
  // ---- per-request work rows (every CTA builds the same table)
  const int per_t = (B + VR_THREADS - 1) / VR_THREADS;
  int32_t my_sum = 0;
  const int32_t tot_rows = p.row_off[B];
  for (int q = 0; q < per_t; ++q) {
    const int r = tid * per_t + q;
    if (r >= B) break;
    const int32_t b0 = p.row_off[r], b1 = p.row_off[r + 1];
    int32_t cnt = 0, len = 0;
    bool valid;
    if (MODE == MODE_TREE) {
      len = b1 - b0;
      valid = b0 >= 0 && len >= 1 && len <= p.max_nodes && b1 <= tot_rows && tot_rows <= p.max_rows;
      cnt = valid ? len : 0;
    } else {
      len = p.verify_len[r];
      valid = len >= 0 && len <= p.L && b0 >= 0 && (int64_t)b0 + len < b1 && b1 <= tot_rows &&
              tot_rows <= p.max_rows;
      cnt = valid ? len + 1 : 0;
      if (valid && MODE == MODE_CHAIN_SAMPLE && p.use_q && p.pm) {
        const uint8_t* pmr = p.pm + (int64_t)r * p.L;
        for (int i = 1; i <= len; ++i)
          if (pmr[i - 1] == 0) {
            if (i <= p.K)
              ++cnt;
            else if (blockIdx.x == 0)
              set_status(p.ws.status, SPEC_DEV_BAD_LENGTH);
          }
      }
    }
    if (!valid && blockIdx.x == 0) set_status(p.ws.status, SPEC_DEV_BAD_LENGTH);
    s_base[r] = b0;
    s_len[r] = valid ? len : -1;
    s_pre[r] = cnt;
    my_sum += cnt;
  }
  // block exclusive scan of the per-thread sums: warp shuffles, then the warp totals
  {
    int32_t x = my_sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t t = __shfl_up_sync(0xFFFFFFFFu, x, o);
      if (lane >= o) x += t;
    }
    if (lane == 31) s_part[warp] = x;
    __syncthreads();
    int32_t before = 0, all = 0;
#pragma unroll
    for (int q = 0; q < VR_WARPS; ++q) {
      const int32_t t = s_part[q];
      if (q < warp) before += t;
      all += t;
    }
    int32_t run = before + x - my_sum;
    for (int q = 0; q < per_t; ++q) {
      const int r = tid * per_t + q;
      if (r >= B) break;
      const int32_t cnt = s_pre[r];
      s_pre[r] = run;
      run += cnt;
    }
    if (tid == 0) s_pre[B] = all;
  }
  __syncthreads();

  // ---- outputs of invalid requests (CTA 0 only)
  if (blockIdx.x == 0) {
    for (int r = warp; r < B; r += VR_WARPS) {
      if (s_len[r] >= 0) continue;
      if (MODE == MODE_TREE) {
        for (int j = lane; j < p.max_nodes; j += 32) {
          p.path[(int64_t)r * p.max_nodes + j] = -1;
          p.out_tokens[(int64_t)r * p.max_nodes + j] = -1;
        }
        if (lane == 0) p.accept_len[r] = -1;
      } else {
        write_invalid_chain(p, r, lane);
      }
    }
  }

  // ---- this warp's contiguous range of chunks (8 KB of one row each)
  constexpr int CH = Vec<DT>::CH;
  const int units = (p.vocab + CH - 1) / CH;  // chunks per row
  const int64_t total = (int64_t)s_pre[B] * units;
  const int64_t nw = (int64_t)gridDim.x * VR_WARPS;
  const int64_t gw = (int64_t)blockIdx.x * VR_WARPS + warp;
  const int64_t lo = gw * total / nw, hi = (gw + 1) * total / nw;
  if (lo >= hi) return;
  const bool vec = p.vec_ok != 0;

  Cursor ic, cc;  // issue and consume cursors
  {
    const int first = (int)(lo / units);
    int a = 0, b = B - 1;  // last r with s_pre[r] <= first
    while (a < b) {
      const int mid = (a + b + 1) >> 1;
      if (s_pre[mid] <= first)
        a = mid;
      else
        b = mid - 1;
    }
    ic.r = cc.r = a;
    ic.item = cc.item = -1;
  }
  // the issue cursor walks (item, chunk) incrementally from lo; it locates a
  // row only when it enters it and then advances its source pointer
  int is_item = (int)(lo / units), is_u = (int)(lo - (int64_t)is_item * units);
  const char* is_src = nullptr;
  auto issue = [&](int s) {
    if (is_src == nullptr) {
      locate<MODE>(p, s_pre, s_base, s_len, is_item, esz, ic);
      is_src = ic.row + (size_t)is_u * CH * esz;
    }
    const uint32_t bytes = (is_u + 1 < units) ? (uint32_t)UB : (uint32_t)((p.vocab - is_u * CH) * esz);
    mbar_arrive_expect_tx(&bars[s], bytes);
    bulk_g2s(stage + (size_t)s * UB, is_src, bytes, &bars[s]);
    is_src += UB;
    if (++is_u == units) {
      is_u = 0;
      ++is_item;
      is_src = nullptr;
    }
  };
  if (vec) {
    if (lane == 0) {
      for (int s = 0; s < ST; ++s) mbar_init(&bars[s], 1);
      fence_mbar_init();
      for (int s = 0; s < ST && lo + s < hi; ++s) issue(s);
    }
    __syncwarp();
  }

  int run_r = -1, run_slot = -1;
  uint32_t run_units = 0;
  unsigned long long run_key = 0ull;
  int bad = 0, aborted = 0;
  int64_t w = lo;

  auto flush_row = [&]() {
    if (MODE != MODE_CHAIN_SAMPLE && run_slot >= 0 && run_key != 0ull && lane == 0)
      atomicMax(&p.ws.rowkey[run_slot], run_key);
  };
  auto flush_request = [&]() {
    if (run_r < 0) return;
    int last = 0;
    if (lane == 0) {
      // release this warp's partials / row keys, acquire everyone else's
      const uint32_t need = (uint32_t)((s_pre[run_r + 1] - s_pre[run_r]) * units);
      const uint32_t old = atomic_add_acq_rel(&p.ws.counter[run_r], run_units);
      last = (old + run_units == need);
    }
    last = __shfl_sync(0xFFFFFFFFu, last, 0);
    if (last) {
      __syncwarp();  // orders every lane after lane 0's acquire
      if (MODE == MODE_TREE)
        finalize_tree(p, run_r, s_base[run_r], s_len[run_r], lane);
      else if (MODE == MODE_CHAIN_GREEDY)
        finalize_chain_greedy<DT>(p, run_r, s_base[run_r], s_len[run_r], lane);
      else
        finalize_chain_sample<DT>(p, run_r, s_base[run_r], s_len[run_r], lane);
      if (lane == 0) p.ws.counter[run_r] = 0u;
    }
  };

  int item = (int)(lo / units), u = (int)(lo - (int64_t)item * units);
  int s = 0;
  uint32_t ph = 0;
  for (; w < hi; ++w) {
    locate<MODE>(p, s_pre, s_base, s_len, item, esz, cc);
    if (cc.slot != run_slot) {
      flush_row();
      run_slot = cc.slot;
      run_key = 0ull;
    }
    if (cc.r != run_r) {
      flush_request();
      run_r = cc.r;
      run_units = 0;
    }
    const int e0 = u * CH;
    const int n_el = min(CH, p.vocab - e0);
    unsigned long long key = 0ull;
    float2 ms[Vec<DT>::SUB];
    if (vec) {
      const bool landed = mbar_wait_bounded(&bars[s], ph, 1u << 22);
      if (!__all_sync(0xFFFFFFFFu, landed)) {  // warp-uniform decision
        aborted = 1;
        break;
      }
      // copy the chunk to registers and refill the stage at once, so that the
      // next copy is in flight while the warp computes
      uint4 v[Vec<DT>::NV];
      vec_load_smem<DT>(stage + (size_t)s * UB, n_el, lane, v);
      __syncwarp();
      if (lane == 0 && w + ST < hi) issue(s);
      if (MODE == MODE_CHAIN_SAMPLE) {
        if (DT == 1) {
          ms[0] = unit_softmax_vec<DT, 0, 8>(v, p.c, bad);
          if (Vec<DT>::SUB > 1) ms[Vec<DT>::SUB - 1] = unit_softmax_vec<DT, 8, 8>(v, p.c, bad);
        } else {
          ms[0] = unit_softmax_vec<DT, 0, 16>(v, p.c, bad);
        }
      } else if (DT == 1) {
        key = chunk_argmax_bf16(v, n_el, lane, bad);
      } else {
        key = unit_argmax_vec<DT>(v, n_el, lane, bad);
      }
    } else {
#pragma unroll
      for (int j = 0; j < Vec<DT>::SUB; ++j) {
        const int e1 = e0 + j * SPEC_UNIT;
        const int n1 = min(SPEC_UNIT, p.vocab - e1);
        if (n1 <= 0) {
          ms[j] = make_float2(-INFINITY, 0.0f);
          continue;
        }
        const void* unit = cc.row + (size_t)e1 * esz;
        if (MODE == MODE_CHAIN_SAMPLE) {
          ms[j] = unit_softmax_scalar<DT>(unit, n1, lane, p.c, bad);
        } else {
          unsigned long long k1 = unit_argmax_scalar<DT>(unit, n1, lane, bad);
          if (k1 != 0ull) {  // rebase to the chunk offset
            const int32_t i1 = argmax_key_index(k1) + j * SPEC_UNIT;
            k1 = (k1 & 0xFFFFFFFF00000000ull) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)i1);
            if (k1 > key) key = k1;
          }
        }
      }
    }
    if (MODE == MODE_CHAIN_SAMPLE) {
      if (lane == 0) {
#pragma unroll
        for (int j = 0; j < Vec<DT>::SUB; ++j) {
          const int uu = u * Vec<DT>::SUB + j;
          if (uu * SPEC_UNIT < p.vocab) __stcg(&p.ws.partial[(int64_t)cc.slot * p.ws.units + uu], ms[j]);
        }
      }
    } else if (key != 0ull) {
      // rebase the chunk offset to the row index; keys of one row fold by max
      const int32_t idx = argmax_key_index(key) + e0;
      const unsigned long long kk =
          (key & 0xFFFFFFFF00000000ull) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)idx);
      if (kk > run_key) run_key = kk;
    }
    ++run_units;
    if (++u == units) {
      u = 0;
      ++item;
    }
    if (++s == ST) {
      s = 0;
      ph ^= 1u;
    }
  }
  if (aborted) {
    // a copy did not land in time: record it, wait (bounded) for every copy this
    // warp still has in flight, and stop without finalizing
    if (lane == 0) {
      set_status(p.ws.status, SPEC_DEV_TIMEOUT);
      for (int64_t x = w; x < hi && x < w + ST; ++x) {
        const int s = (int)((x - lo) % ST);
        mbar_wait_bounded(&bars[s], (uint32_t)(((x - lo) / ST) & 1), 1u << 22);
      }
    }
    __syncwarp();
    return;
  }
  flush_row();
  flush_request();
  if (bad && lane == 0) set_status(p.ws.status, SPEC_DEV_NONFINITE);
}

// ------------------------------------------------------------------ draw from max(0, p - q)
template <int DT>
__global__ void __launch_bounds__(SPEC_CTA_THREADS) resample_kernel(VerifyParams p) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int units = p.units;
  const int64_t total = (int64_t)p.batch * units;
  const int64_t nwarps = (int64_t)gridDim.x * SPEC_WARPS_PER_CTA;
  const size_t esz = DT == 1 ? 2 : 4;
  const bool vec = p.vec_ok != 0;
  for (int64_t w = (int64_t)blockIdx.x * SPEC_WARPS_PER_CTA + warp; w < total; w += nwarps) {
    const int r = (int)(w / units);
    const int u = (int)(w - (int64_t)r * units);
    // the whole record in one round trip (four 16-byte loads)
    Record rec;
    {
      const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const Record*>(p.ws.record) + r);
      uint4* dst = reinterpret_cast<uint4*>(&rec);
#pragma unroll
      for (int q = 0; q < 4; ++q) dst[q] = __ldcg(src + q);
    }
    if (!rec.flag) continue;
    const void* prow = static_cast<const char*>(p.logits) + (int64_t)rec.prow * p.vocab * esz;
    const void* qrow = static_cast<const char*>(p.draft) +
                       ((int64_t)r * p.K + rec.pos - 1) * p.vocab * esz;
    const float ip = 1.0f / rec.sp, iq = 1.0f / rec.sq;
    const float mpc = rec.mp * p.c, mqc = rec.mq * p.c;
    auto resid = [&](const float* vp, const float* vq, int j) -> float {
      const float a = vp[j] == -INFINITY ? 0.0f : ex2(fmaf(vp[j], p.c, -mpc)) * ip;
      const float b = vq[j] == -INFINITY ? 0.0f : ex2(fmaf(vq[j], p.c, -mqc)) * iq;
      return a > b ? a - b : 0.0f;
    };
    {
      const int e0 = u * SPEC_UNIT, n_el = min(SPEC_UNIT, p.vocab - e0);
      float vp[64], vq[64];
      load_unit_contig<DT>(prow, e0, n_el, vec, lane, vp);
      load_unit_contig<DT>(qrow, e0, n_el, vec, lane, vq);
      float a0 = 0.0f, a1 = 0.0f;
#pragma unroll
      for (int j = 0; j < 64; j += 2) {
        a0 += resid(vp, vq, j);
        a1 += resid(vp, vq, j + 1);
      }
      const float ws = warp_sum(a0 + a1);
      if (lane == 0) __stcg(&p.ws.partial2[(int64_t)r * p.ws.units + u], (double)ws);
    }
    int last = 0;
    if (lane == 0) {
      __threadfence();
      const uint32_t old = atomicAdd(&p.ws.counter2[r], 1u);
      last = (old + 1u == (uint32_t)units);
    }
    last = __shfl_sync(0xFFFFFFFFu, last, 0);
    if (!last) continue;
    __threadfence();
    // the residual mass; at or below 1e-30 the draw falls back to p
    const int pslot = rec.prow;
    auto w_res = [&](int uu) -> float { return (float)__ldcg(&p.ws.partial2[(int64_t)r * p.ws.units + uu]); };
    auto w_p = [&](int uu) -> float {
      const float2 t = __ldcg(&p.ws.partial[(int64_t)pslot * p.ws.units + uu]);
      if (t.x == -INFINITY) return 0.0f;
      return t.y * ex2((t.x - rec.mp) * p.c) * ip;
    };
    Crossing cr = find_unit(units, rec.u2, lane, w_res);
    const bool fallback = !(cr.total > 1e-30f);
    if (fallback) cr = find_unit(units, rec.u2, lane, w_p);
    const int e0 = cr.unit * SPEC_UNIT, n_el = min(SPEC_UNIT, p.vocab - e0);
    float vp[64], vq[64], rr[64];
    load_unit_contig<DT>(prow, e0, n_el, vec, lane, vp);
    load_unit_contig<DT>(qrow, e0, n_el, vec, lane, vq);
#pragma unroll
    for (int j = 0; j < 64; ++j)
      rr[j] = fallback ? (vp[j] == -INFINITY ? 0.0f : ex2(fmaf(vp[j], p.c, -mpc)) * ip) : resid(vp, vq, j);
    float r_at;
    const int pick = find_in_unit(rr, cr.before, cr.t, lane, &r_at);
    if (lane == 0) {
      p.out_tokens[(int64_t)r * (p.L + 1) + rec.pos - 1] = e0 + pick;
      if (p.dbg_resid) p.dbg_resid[r] = r_at / cr.total;
      Record* wr = reinterpret_cast<Record*>(p.ws.record) + r;
      wr->flag = 0;
      p.ws.counter2[r] = 0u;
    }
  }
}

// ------------------------------------------------------------------ probabilistic drafting
// y_k ~ softmax(z_k / T) for the drafter's rows (Hybrid Spark sec. 4.5, App. H).
// One pass over each row: per 8 KB chunk, (max, sum of 2^((z - max) log2e / T))
// per 2048-entry unit into the workspace partials -- the slots the verification
// kernel uses for the same q rows -- and the warp that completes a row draws
// from it: the crossing unit from the units' weights, then the crossing entry
// inside that unit (a second read of one 4-8 KB unit).  The uniform is word 0
// of Philox counter (r, 0x40000000 + k, lo32(step), hi32(step)), key
// (lo32(seed), hi32(seed)), a counter domain apart from verification's.
template <int DT>
__device__ void draw_draft(const VerifyParams& p, int row, int r, int k, int slot, int lane) {
  // the row's unit partials, lane l holding units [per l, per l + per) (the
  // layout find_unit walks), loaded once for the row max and the weights
  const int per = (p.units + 31) / 32, u0 = lane * per;
  const float2* pr = &p.ws.partial[(int64_t)slot * p.ws.units];
  float2 t4[4];
#pragma unroll
  for (int q = 0; q < 4; ++q)
    t4[q] = (q < per && u0 + q < p.units) ? __ldcg(&pr[u0 + q]) : make_float2(-INFINITY, 0.0f);
  float lm = fmaxf(fmaxf(t4[0].x, t4[1].x), fmaxf(t4[2].x, t4[3].x));
  for (int q = 4; q < per; ++q)
    if (u0 + q < p.units) lm = fmaxf(lm, __ldcg(&pr[u0 + q]).x);
  const float m = warp_max(lm);
  uint32_t o[4];
  philox4x32_10((uint32_t)r, 0x40000000u + (uint32_t)(k + 1), (uint32_t)p.step, (uint32_t)(p.step >> 32),
                (uint32_t)p.seed, (uint32_t)(p.seed >> 32), o);
  const float u = (float)(o[0] >> 8) * (1.0f / 16777216.0f);
  const char* base = static_cast<const char*>(p.draft) + (int64_t)row * p.vocab * (DT == 1 ? 2 : 4);
  int y = 0;
  float q_at = 0.0f;
  float total = 0.0f;
  if (m != -INFINITY) {
    auto w_plain = [&](int uu) -> float {
      const int q = uu - u0;
      const float2 t = q == 0 ? t4[0] : q == 1 ? t4[1] : q == 2 ? t4[2] : q == 3 ? t4[3] : __ldcg(&pr[uu]);
      if (t.x == -INFINITY) return 0.0f;
      return t.y * ex2((t.x - m) * p.c);
    };
    const Crossing cr = find_unit(p.units, u, lane, w_plain);
    total = cr.total;
    float v[64];
    const int e0 = cr.unit * SPEC_UNIT;
    const int n_el = min(SPEC_UNIT, p.vocab - e0);
    load_unit_contig<DT>(base, e0, n_el, p.vec_ok != 0, lane, v);
    const float mc = m * p.c;
#pragma unroll
    for (int j = 0; j < 64; ++j) v[j] = (v[j] == -INFINITY) ? 0.0f : ex2(fmaf(v[j], p.c, -mc));
    const int pick = find_in_unit(v, cr.before, cr.t, lane, &q_at);
    y = e0 + pick;
  }
  if (lane == 0) {
    p.out_tokens[row] = y;
    if (p.dbg_u) p.dbg_u[row] = u;
    if (p.dbg_resid) p.dbg_resid[row] = total > 0.0f ? q_at / total : 0.0f;
  }
}

template <int DT>
__global__ void __launch_bounds__(SPEC_CTA_THREADS) sample_drafts_kernel(VerifyParams p) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int CH = Vec<DT>::CH, SUB = Vec<DT>::SUB;
  const int chunks = (p.vocab + CH - 1) / CH;
  const int rows = p.batch * p.K;
  const int64_t total = (int64_t)rows * chunks;
  const int64_t nwarps = (int64_t)gridDim.x * SPEC_WARPS_PER_CTA;
  const size_t esz = DT == 1 ? 2 : 4;
  const bool vec = p.vec_ok != 0;
  int bad = 0;
  for (int64_t w = (int64_t)blockIdx.x * SPEC_WARPS_PER_CTA + warp; w < total; w += nwarps) {
    const int row = (int)(w / chunks), ch = (int)(w - (int64_t)row * chunks);
    const int r = row / p.K, k = row - r * p.K;  // position k + 1
    const int slot = q_slot_of(p, r, k + 1);
    const char* base = static_cast<const char*>(p.draft) + (int64_t)row * p.vocab * esz;
    const int e0 = ch * CH, n_el = min(CH, p.vocab - e0);
    float2 ms[SUB];
    if (vec) {
      uint4 v[Vec<DT>::NV];
      vec_load_global<DT>(base + (size_t)e0 * esz, n_el, lane, v);
      if (DT == 1) {
        ms[0] = unit_softmax_vec<DT, 0, 8>(v, p.c, bad);
        if (SUB > 1) ms[SUB - 1] = unit_softmax_vec<DT, 8, 8>(v, p.c, bad);
      } else {
        ms[0] = unit_softmax_vec<DT, 0, 16>(v, p.c, bad);
      }
    } else {
#pragma unroll
      for (int j = 0; j < SUB; ++j) {
        const int e1 = e0 + j * SPEC_UNIT;
        const int n1 = min(SPEC_UNIT, p.vocab - e1);
        ms[j] = n1 <= 0 ? make_float2(-INFINITY, 0.0f)
                        : unit_softmax_scalar<DT>(base + (size_t)e1 * esz, n1, lane, p.c, bad);
      }
    }
    int last = 0;
    if (lane == 0) {
#pragma unroll
      for (int j = 0; j < SUB; ++j) {
        const int uu = ch * SUB + j;
        if (uu * SPEC_UNIT < p.vocab) __stcg(&p.ws.partial[(int64_t)slot * p.ws.units + uu], ms[j]);
      }
      // release this chunk's partials, acquire the row's others
      const uint32_t old = atomic_add_acq_rel(&p.ws.counter3[row], 1u);
      last = (old + 1u == (uint32_t)chunks);
    }
    last = __shfl_sync(0xFFFFFFFFu, last, 0);
    if (last) {
      __syncwarp();  // orders every lane after lane 0's acquire
      if (lane == 0) p.ws.counter3[row] = 0u;
      draw_draft<DT>(p, row, r, k, slot, lane);
    }
  }
  if (bad && lane == 0) set_status(p.ws.status, SPEC_DEV_NONFINITE);
}

}  // namespace spec

// ---------------------------------------------------------------------------
// host launchers (called from api.cu)
// ---------------------------------------------------------------------------
namespace {

template <typename Kern>
int grid_for(Kern k, size_t smem, int num_sms) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, SPEC_CTA_THREADS, smem) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  return per_sm * num_sms;
}

template <int DT, int MODE>
cudaError_t launch_rows(const spec::VerifyParams& p, int num_sms, cudaStream_t stream) {
  using V = spec::Vec<DT>;
  const size_t smem = (size_t)VR_WARPS * V::STAGES * (V::BYTES + 8) +
                      (size_t)(3 * p.batch + 1) * sizeof(int32_t);
  auto k = spec::verify_rows_kernel<DT, MODE>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  // one CTA per SM: the shared-memory rings hold the bytes in flight
  k<<<num_sms, VR_THREADS, smem, stream>>>(p);
  return cudaGetLastError();
}

template <int DT>
cudaError_t launch_resample(const spec::VerifyParams& p, int num_sms, cudaStream_t stream) {
  auto k = spec::resample_kernel<DT>;
  static int cached_grid = 0;
  if (cached_grid == 0) cached_grid = grid_for(k, 0, num_sms);
  int64_t need = ((int64_t)p.batch * p.units + SPEC_WARPS_PER_CTA - 1) / SPEC_WARPS_PER_CTA;
  int grid = (int)(need < cached_grid ? need : cached_grid);
  if (grid < 1) grid = 1;
  k<<<grid, SPEC_CTA_THREADS, 0, stream>>>(p);
  return cudaGetLastError();
}

spec::WsView ws_view(const spec_workspace* ws) {
  spec::WsView v;
  char* b = static_cast<char*>(ws->base);
  v.status = reinterpret_cast<uint32_t*>(b);
  v.counter = reinterpret_cast<uint32_t*>(b + ws->off_counter);
  v.counter2 = reinterpret_cast<uint32_t*>(b + ws->off_counter2);
  v.counter3 = reinterpret_cast<uint32_t*>(b + ws->off_counter3);
  v.record = reinterpret_cast<unsigned char*>(b + ws->off_record);
  v.rowkey = reinterpret_cast<unsigned long long*>(b + ws->off_rowkey);
  v.partial = reinterpret_cast<float2*>(b + ws->off_partial);
  v.partial2 = reinterpret_cast<double*>(b + ws->off_partial2);
  v.units = ws->units;
  v.max_rows = ws->max_rows;
  v.max_batch = ws->max_batch;
  v.K = ws->K;
  return v;
}

}  // namespace

extern "C" cudaError_t spec_launch_verify_chain(
    int32_t batch, int32_t vocab, int32_t dtype, const void* logits, const int32_t* row_off,
    const void* draft, int32_t K, const int32_t* chain, int32_t L, const int32_t* verify_len,
    const uint8_t* pm, float temperature, uint64_t seed, uint64_t step, int32_t* out_tokens,
    int32_t* n_accepted, int32_t* n_emitted, float* dbg_ratio, float* dbg_u, float* dbg_resid,
    const spec_workspace* ws, int num_sms, cudaStream_t stream) {
  spec::VerifyParams p = {};
  p.batch = batch;
  p.vocab = vocab;
  p.logits = logits;
  p.row_off = row_off;
  p.max_rows = ws->max_rows;
  p.draft = draft;
  p.K = draft ? K : 0;
  p.chain = chain;
  p.L = L;
  p.verify_len = verify_len;
  p.pm = pm;
  const bool greedy = !(temperature > 0.0f);
  p.use_q = (!greedy && draft != nullptr && pm != nullptr) ? 1 : 0;
  p.c = greedy ? 0.0f : (float)(1.4426950408889634 / (double)temperature);
  p.seed = seed;
  p.step = step;
  p.out_tokens = out_tokens;
  p.n_accepted = n_accepted;
  p.n_emitted = n_emitted;
  p.dbg_ratio = dbg_ratio;
  p.dbg_u = dbg_u;
  p.dbg_resid = dbg_resid;
  p.units = (vocab + SPEC_UNIT - 1) / SPEC_UNIT;
  const size_t esz = dtype == SPEC_BF16 ? 2 : 4;
  p.vec_ok = (((size_t)vocab * esz) % 16 == 0 && (reinterpret_cast<uintptr_t>(logits) & 15u) == 0 &&
              (draft == nullptr || (reinterpret_cast<uintptr_t>(draft) & 15u) == 0))
                 ? 1
                 : 0;
  p.ws = ws_view(ws);
  if (batch == 0) return cudaSuccess;
  cudaError_t e;
  if (dtype == SPEC_BF16)
    e = greedy ? launch_rows<1, spec::MODE_CHAIN_GREEDY>(p, num_sms, stream)
               : launch_rows<1, spec::MODE_CHAIN_SAMPLE>(p, num_sms, stream);
  else
    e = greedy ? launch_rows<0, spec::MODE_CHAIN_GREEDY>(p, num_sms, stream)
               : launch_rows<0, spec::MODE_CHAIN_SAMPLE>(p, num_sms, stream);
  if (e != cudaSuccess || !p.use_q) return e;
  return dtype == SPEC_BF16 ? launch_resample<1>(p, num_sms, stream) : launch_resample<0>(p, num_sms, stream);
}

extern "C" cudaError_t spec_launch_verify_tree(int32_t batch, int32_t vocab, int32_t dtype,
                                               const void* logits, const int32_t* node_off,
                                               const int32_t* tok, const int32_t* parent,
                                               int32_t max_nodes, int32_t* path, int32_t* accept_len,
                                               int32_t* out_tokens, const spec_workspace* ws,
                                               int num_sms, cudaStream_t stream) {
  spec::VerifyParams p = {};
  p.batch = batch;
  p.vocab = vocab;
  p.logits = logits;
  p.row_off = node_off;
  p.max_rows = ws->max_rows;
  p.tok = tok;
  p.parent = parent;
  p.max_nodes = max_nodes;
  p.path = path;
  p.accept_len = accept_len;
  p.out_tokens = out_tokens;
  p.units = (vocab + SPEC_UNIT - 1) / SPEC_UNIT;
  const size_t esz = dtype == SPEC_BF16 ? 2 : 4;
  p.vec_ok = (((size_t)vocab * esz) % 16 == 0 && (reinterpret_cast<uintptr_t>(logits) & 15u) == 0) ? 1 : 0;
  p.ws = ws_view(ws);
  if (batch == 0) return cudaSuccess;
  return dtype == SPEC_BF16 ? launch_rows<1, spec::MODE_TREE>(p, num_sms, stream)
                            : launch_rows<0, spec::MODE_TREE>(p, num_sms, stream);
}

extern "C" cudaError_t spec_launch_sample_drafts(int32_t batch, int32_t K, int32_t vocab, int32_t dtype,
                                                 const void* draft_logits, float temperature, uint64_t seed,
                                                 uint64_t step, int32_t* y, float* dbg_u, float* dbg_q,
                                                 const spec_workspace* ws, int num_sms, cudaStream_t stream) {
  spec::VerifyParams p = {};
  p.batch = batch;
  p.vocab = vocab;
  p.max_rows = ws->max_rows;
  p.draft = draft_logits;
  p.K = K;
  p.c = (float)(1.4426950408889634 / (double)temperature);
  p.seed = seed;
  p.step = step;
  p.out_tokens = y;
  p.dbg_u = dbg_u;
  p.dbg_resid = dbg_q;
  p.units = (vocab + SPEC_UNIT - 1) / SPEC_UNIT;
  const size_t esz = dtype == SPEC_BF16 ? 2 : 4;
  p.vec_ok = (((size_t)vocab * esz) % 16 == 0 && (reinterpret_cast<uintptr_t>(draft_logits) & 15u) == 0) ? 1 : 0;
  p.ws = ws_view(ws);
  if (batch == 0) return cudaSuccess;
  const int ch = dtype == SPEC_BF16 ? spec::Vec<1>::CH : spec::Vec<0>::CH;
  const int64_t chunks = (int64_t)batch * K * ((vocab + ch - 1) / ch);
  const int64_t want = (chunks + SPEC_WARPS_PER_CTA - 1) / SPEC_WARPS_PER_CTA;
  const int grid = (int)(want < (int64_t)num_sms * 8 ? want : (int64_t)num_sms * 8);
  if (dtype == SPEC_BF16)
    spec::sample_drafts_kernel<1><<<grid, SPEC_CTA_THREADS, 0, stream>>>(p);
  else
    spec::sample_drafts_kernel<0><<<grid, SPEC_CTA_THREADS, 0, stream>>>(p);
  return cudaGetLastError();
}
