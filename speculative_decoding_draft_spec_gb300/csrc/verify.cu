// verify.cu -- steps 3 and 4 of the round: chain verification and greedy tree
// verification over full-vocabulary logit rows, and the drafter's
// probabilistic tokens (a draw per draft row).
//
// Chain (Hybrid Spark sec. 2, App. H; the fixed-cost parallel drafter page's
// verification rule): accept y_i iff u_i < min(1, p_i(y_i)/q_i(y_i)), q a
// point mass for greedy / n-gram drafts; at the first rejection draw from
// norm(max(0, p_i - q_i)); after all acceptances draw a bonus from p_{ell+1};
// T = 0 accepts iff y_i = argmax.  r accepted => r + 1 tokens.
// Tree (AdaSpark sec. 2.2): a node is accepted iff its token equals the argmax
// at its parent's row and its parent is accepted; commit the path and the
// argmax after it.
// Drafting (Hybrid Spark sec. 4.5, App. H): y_k ~ softmax(z_k / T) for each
// draft row, by inverse CDF at a Philox uniform.
//
// GB300 layout.  The HBM-bound part is one pass over every row.  One CTA per
// SM, 12 warps each; the work is the sequence of 8 KB chunks of the rows (4096
// bf16 / 2048 fp32 entries) in (request, row, chunk) order, and every warp
// takes an equal contiguous range of it.  Each warp streams its range through
// its own 8 KB shared-memory stage, filled by one-dimensional bulk async
// copies (completion on an mbarrier, bounded wait): it moves a landed chunk
// into registers and refills the stage at once, so one copy per warp is in
// flight (longer memory queues widen the spread of the warps' finish times).
// Per chunk a warp produces
//   greedy / tree rows: a packed 64-bit (ordered value, ~index) key; keys of
//                 one row fold in registers and reach the row's workspace key
//                 with one atomicMax per run of the row (largest value, lowest
//                 index);
//   sampled rows: the chunk's (max, sum of 2^((z - max) log2e / T)) in the
//                 workspace, and the logit at the row's draft token when the
//                 chunk holds it.
// Each request (each draft row, when drafting) has an arrival counter; the
// warp that completes its last chunk (acquire-release atomic, no waiting)
// finalizes it in an 8 KB scratch of its own beside its stage: the request's
// partial rows arrive there by one bulk copy each, so merging the row
// normalisers, reading p(y) and q(y) and locating a draw's chunk take one
// memory round trip, and a draw's chunk is then walked in shared memory.  A
// draw from max(0, p - q) needs a second pass over two rows once both
// normalisers are known; those requests are finished by resample_kernel, one
// CTA per (request, chunk).
#include <cuda_bf16.h>

#include "common.cuh"

namespace spec {

enum { MODE_CHAIN_GREEDY = 0, MODE_CHAIN_SAMPLE = 1, MODE_TREE = 2, MODE_DRAFT = 3 };

#define VR_WARPS 12
#define VR_THREADS (32 * VR_WARPS)
#define VR_STAGE 8192            // bytes per stage: one chunk (one copy in flight per warp)
#define VR_BARS 2                // per warp: the stage's, and the finalizer scratch's
// shared memory of one warp: its stage, then (sampled modes) the finalizer's scratch
#define VR_WBUF(MODE) (VR_STAGE * ((MODE) == ::spec::MODE_CHAIN_SAMPLE || (MODE) == ::spec::MODE_DRAFT ? 2 : 1))
#define RS_THREADS 256           // resample_kernel: one CTA per (request, chunk)
#define SPEC_WAIT_POLLS (1u << 22)

struct VerifyParams {
  int32_t batch, vocab;
  const void* logits;      // target logits (chain) or tree logits
  const int32_t* row_off;  // chain: row_off [batch+1]; tree: node_off [batch+1]
  int32_t max_rows;
  int32_t qbase;  // partial slot of draft row (r, i) = qbase + r K + i - 1
  const void* draft;  // [batch x K x vocab] or null
  int32_t K;
  const int32_t* chain;
  int32_t L;
  const int32_t* verify_len;
  const uint8_t* pm;
  int32_t use_q;  // draft logits present and T > 0
  int32_t reuse_q;  // the draft rows' partials and spare entries come from the drafting call: not streamed
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
  int32_t nch;      // chunks per row: ceil(vocab / entries per chunk)
  int32_t rowf;     // float2 entries of a staged partial row: nch + 1 (the spare), rounded up to even
  int32_t pstride;  // float2 entries between partial rows in the workspace (>= rowf)
  int32_t vec_ok;   // every row starts on a 16-byte boundary
  uint64_t m_nw;    // floor(2^32 / d) + 1 for d = the grid's warps (division by a multiply-high)
  uint64_t m_nch;   // the same for d = nch
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

__device__ __forceinline__ float2* partial_row(const VerifyParams& p, int slot) {
  return p.ws.partial + (int64_t)slot * p.pstride;
}
// the draft row (request r, 1-based position i) that carries q_i: its workspace slot
// n / d for n < 2^31 from m = floor(2^32 / d) + 1: m d exceeds 2^32 by at
// most d, so the multiply-high is the quotient or one more (n < 2^31 keeps the
// excess below 1/2), and one test corrects it
__device__ __forceinline__ uint32_t udiv(uint32_t n, uint32_t d, uint64_t m) {
  const uint32_t q = (uint32_t)(((uint64_t)n * m) >> 32);
  return q * d > n ? q - 1u : q;
}

__device__ __forceinline__ int q_slot_of(const VerifyParams& p, int r, int i) {
  return p.qbase + r * p.K + (i - 1);
}
// index of the n-th (0-based) set bit of m
__device__ __forceinline__ int nth_bit(uint32_t m, int n) {
  for (int t = 0; t < n; ++t) m &= m - 1u;
  return __ffs(m) - 1;
}

// ------------------------------------------------------------------ loading
// strided layout: lane-interleaved 16-byte vectors (coalesced); element j of
// a lane sits at unit offset idx_strided<DT>(lane, j)
template <int DT>
__device__ __forceinline__ int idx_strided(int lane, int j, bool vec) {
  if (!vec) return lane + 32 * j;
  if (DT == 1) return 8 * (lane + 32 * (j >> 3)) + (j & 7);
  return 4 * (lane + 32 * (j >> 2)) + (j & 3);
}

// 64 values of one 2048-entry unit in scalar loads (element j of a lane at
// offset lane + 32 j), missing entries = -inf; for rows that are not 16-byte
// aligned
template <int DT>
__device__ __forceinline__ void load_unit(const void* row, int e0, int n_el, bool vec, int lane, float v[64]) {
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
  static constexpr int BYTES = VR_STAGE;       // bytes per chunk (one stage)
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


// ------------------------------------------------------------------ draws
// Inverse CDF over chunk weights (chunk order) at the fraction u of their
// total: the chunk holding the crossing of t = u * total, the weight before
// it, the total and t.  Lane l holds the weights of chunks [per l, per l +
// per) in wl (per <= 8), so lane order is chunk order; the sums run in fp32.
struct Crossing {
  int unit;      // the crossing chunk
  float before;  // weight of the chunks before it; -1: t at or above the total (take the last entry)
  float total;
  float t;
};

__device__ __forceinline__ Crossing find_chunk(const float (&wl)[8], int per, float u, int lane) {
  float lsum = 0.0f;
  int last_q = -1;
#pragma unroll
  for (int q = 0; q < 8; ++q)
    if (q < per) {
      lsum += wl[q];
      if (wl[q] > 0.0f) last_q = q;
    }
  const float incl = warp_incl_scan(lsum);
  const float excl = incl - lsum;
  Crossing c;
  c.total = __shfl_sync(0xFFFFFFFFu, incl, 31);
  c.t = u * c.total;
  const unsigned hit = __ballot_sync(0xFFFFFFFFu, incl > c.t && lsum > 0.0f);
  if (hit) {
    const int src = __ffs(hit) - 1;
    int unit = -1;
    float before = 0.0f, run = excl, wlast = 0.0f;
#pragma unroll
    for (int q = 0; q < 8; ++q)
      if (q < per) {
        if (unit < 0 && wl[q] > 0.0f && run + wl[q] > c.t) {
          unit = per * lane + q;
          before = run;
        }
        run += wl[q];
        if (q == last_q) wlast = wl[q];
      }
    if (unit < 0) {  // rounding inside the lane: its last chunk with weight
      unit = per * lane + last_q;
      before = incl - wlast;
    }
    c.unit = __shfl_sync(0xFFFFFFFFu, unit, src);
    c.before = __shfl_sync(0xFFFFFFFFu, before, src);
  } else {  // t at or above the total (rounding): the last chunk with weight
    const unsigned has = __ballot_sync(0xFFFFFFFFu, last_q >= 0);
    const int src = has ? 31 - __clz(has) : 0;
    const int lp = __shfl_sync(0xFFFFFFFFu, per * lane + last_q, src);
    c.unit = has ? lp : 0;
    c.before = -1.0f;
  }
  return c;
}

// A chunk staged in shared memory, seen as 16 steps of 32 x PER consecutive
// entries (32 vectors of 16 bytes each).  Lanes 2k and 2k + 1 sum the two
// halves of step k, 16 vectors each, in a rolled loop whose reads are rotated
// by k (odd lanes by k + 4) so that each quarter-warp's 16-byte reads fall in
// distinct banks; one pair shuffle then gives the step totals, and the
// crossing step is read once more as vector `lane` of that step.  Entries that
// take no part hold -inf in the stage (a chunk's tail past the row, an entry
// left out), so no entry carries a test.  The finalizing warp runs this once,
// alone on its scheduler: compact code (a rolled loop, few cold instruction
// lines) with overlapping exponentials inside an iteration is what counts.

// entry i (< PER) of a vector
template <int DT>
__device__ __forceinline__ float vec_entry(const uint4& x, int i) {
  constexpr int EW = DT == 1 ? 2 : 1;  // entries per word
  const int q = i / EW;
  const uint32_t w = q == 0 ? x.x : q == 1 ? x.y : q == 2 ? x.z : x.w;
  return DT == 1 ? ((i & 1) ? bf16_hi(w) : bf16_lo(w)) : __uint_as_float(w);
}

// the weights 2^(z c - mc) of a vector, summed as a tree
template <int DT>
__device__ __forceinline__ float vec_weight(const uint4& x, float mc, float c) {
  constexpr int PER = Vec<DT>::PER;
  float t[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) t[i] = ex2(fmaf(vec_entry<DT>(x, i), c, -mc));  // 2^-inf = +0
#pragma unroll
  for (int h = PER / 2; h > 0; h >>= 1)
#pragma unroll
    for (int i = 0; i < h; ++i) t[i] += t[i + h];
  return t[0];
}

// the lane's half-step sum (lane 2k + h: half h of step k)
template <int DT>
__device__ __forceinline__ float half_step_sum(const unsigned char* buf, float mc, float c, int lane) {
  const int k = lane >> 1, h = lane & 1;
  const uint4* base = reinterpret_cast<const uint4*>(buf) + 32 * k + 16 * h;
  const int rot = k + 4 * h;
  float s0 = 0.0f, s1 = 0.0f;
#pragma unroll 2
  for (int j = 0; j < 16; j += 2) {
    s0 += vec_weight<DT>(base[(j + rot) & 15], mc, c);
    s1 += vec_weight<DT>(base[(j + 1 + rot) & 15], mc, c);
  }
  return s0 + s1;
}

// the warp total of a staged chunk's weights
template <int DT>
__device__ __forceinline__ float chunk_sum(const unsigned char* buf, float mc, float c, int lane) {
  return warp_sum(half_step_sum<DT>(buf, mc, c, lane));
}

// Inverse CDF inside a staged chunk: the first entry whose running sum from
// `before` exceeds t (before < 0, or no crossing after rounding: the last
// entry with weight), by the step whose running total crosses it and then the
// entry inside that step.  Weights 2^(z c - mc).  Returns the entry and *w_at
// its weight.
template <int DT>
__device__ int chunk_draw(const unsigned char* buf, int lane, float before, float t, float* w_at, float mc, float c) {
  constexpr int PER = Vec<DT>::PER;
  const float hs = half_step_sum<DT>(buf, mc, c, lane);
  const float stot = hs + __shfl_xor_sync(0xFFFFFFFFu, hs, 1);
  const float st = __shfl_sync(0xFFFFFFFFu, stot, (2 * lane) & 31);
  const float sk = lane < 16 ? st : 0.0f;  // lane k: step k's total
  const float incl = warp_incl_scan(sk);
  const float tl = before < 0.0f ? INFINITY : t - before;
  const unsigned has = __ballot_sync(0xFFFFFFFFu, sk > 0.0f);
  const unsigned hit = __ballot_sync(0xFFFFFFFFu, incl > tl && sk > 0.0f);  // none for tl = INFINITY
  int ks;
  float t2;
  if (hit) {
    ks = __ffs(hit) - 1;
    t2 = tl - __shfl_sync(0xFFFFFFFFu, incl - sk, ks);
  } else {
    ks = has ? 31 - __clz(has) : 0;
    t2 = INFINITY;
  }
  const uint4 x = reinterpret_cast<const uint4*>(buf)[32 * ks + lane];
  const int e = PER * (32 * ks + lane);
  float wv[PER], ls = 0.0f;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    wv[i] = ex2(fmaf(vec_entry<DT>(x, i), c, -mc));
    ls += wv[i];
  }
  const float inc2 = warp_incl_scan(ls);
  const unsigned hit2 = __ballot_sync(0xFFFFFFFFu, inc2 > t2 && ls > 0.0f);
  int pick = -1, lp = -1;
  float wp = 0.0f, lw = 0.0f, run = inc2 - ls;
#pragma unroll
  for (int i = 0; i < PER; ++i)
    if (wv[i] > 0.0f) {
      run += wv[i];
      if (pick < 0 && run > t2) {
        pick = e + i;
        wp = wv[i];
      }
      lp = e + i;
      lw = wv[i];
    }
  int src;
  if (hit2) {
    src = __ffs(hit2) - 1;
    if (pick < 0) {  // rounding inside the lane: its last entry with weight
      pick = lp;
      wp = lw;
    }
  } else {
    const unsigned h2 = __ballot_sync(0xFFFFFFFFu, lp >= 0);
    src = h2 ? 31 - __clz(h2) : 0;
    pick = lp;
    wp = lw;
  }
  pick = __shfl_sync(0xFFFFFFFFu, pick, src);
  *w_at = __shfl_sync(0xFFFFFFFFu, wp, src);
  return pick < 0 ? 0 : pick;
}

// entry i of a staged chunk set to -inf (returns its bits) or back to `bits`
template <int DT>
__device__ __forceinline__ uint32_t stage_entry_swap(unsigned char* buf, int i, uint32_t bits) {
  if (DT == 1) {
    uint16_t* q = reinterpret_cast<uint16_t*>(buf) + i;
    const uint32_t old = *q;
    *q = (uint16_t)bits;
    return old;
  }
  uint32_t* q = reinterpret_cast<uint32_t*>(buf) + i;
  const uint32_t old = *q;
  *q = bits;
  return old;
}

// ------------------------------------------------------------------ finalizer scratch
// 8 KB of a warp's shared memory beside its stage, filled by bulk copies that
// complete on the warp's second mbarrier.
struct Scratch {
  unsigned char* buf;
  uint64_t* bar;
  uint32_t phase;
  int dead;  // a copy did not land in time: the scratch is not used again
};

// wait for the scratch's copies; false (SPEC_DEV_TIMEOUT set) when the bound ran out
__device__ __forceinline__ bool scratch_wait(Scratch& sc, uint32_t* status, int lane) {
  const bool ok = mbar_wait_bounded(sc.bar, sc.phase, SPEC_WAIT_POLLS);
  sc.phase ^= 1u;
  if (__all_sync(0xFFFFFFFFu, ok)) return true;
  if (lane == 0) set_status(status, SPEC_DEV_TIMEOUT);
  sc.dead = 1;
  return false;
}

// n <= 32 partial rows into the scratch (row j from slot slot_of(j), rowf
// float2 each): one bulk copy per run of rows whose slots are consecutive (a
// request's target rows are one run, its draft rows runs of consecutive
// positions), issued by the run's first lane; stage_rows_issue returns at once
// (scratch_wait completes it), stage_rows waits
template <typename SlotFn>
__device__ __forceinline__ void stage_rows_issue(const VerifyParams& p, Scratch& sc, int n, SlotFn slot_of,
                                                 int lane) {
  const uint32_t rb = (uint32_t)p.rowf * 8u;
  fence_proxy_async();
  if (lane == 0) mbar_arrive_expect_tx(sc.bar, rb * (uint32_t)n);
  __syncwarp();
  const int sl = lane < n ? slot_of(lane) : 0;
  const int prev = __shfl_up_sync(0xFFFFFFFFu, sl, 1);
  const bool start = lane < n && (lane == 0 || sl != prev + 1);
  const unsigned starts = __ballot_sync(0xFFFFFFFFu, start);
  if (start) {
    const unsigned later = lane < 31 ? starts & ~((2u << lane) - 1u) : 0u;
    const int end = later ? __ffs(later) - 1 : n;
    bulk_g2s(sc.buf + (size_t)lane * rb, partial_row(p, sl), rb * (uint32_t)(end - lane), sc.bar);
  }
}
template <typename SlotFn>
__device__ __forceinline__ bool stage_rows(const VerifyParams& p, Scratch& sc, int n, SlotFn slot_of, int lane) {
  stage_rows_issue(p, sc, n, slot_of, lane);
  return scratch_wait(sc, p.ws.status, lane);
}

// the n_el entries of a row from entry e0 into the scratch (one chunk)
template <int DT>
__device__ __forceinline__ bool stage_chunk(const VerifyParams& p, Scratch& sc, const void* row, int e0, int n_el,
                                            int lane) {
  constexpr int ESZ = DT == 1 ? 2 : 4;
  constexpr int CH = Vec<DT>::CH;
  if (p.vec_ok) {
    if (lane == 0) {
      mbar_arrive_expect_tx(sc.bar, (uint32_t)(n_el * ESZ));
      bulk_g2s(sc.buf, static_cast<const char*>(row) + (size_t)e0 * ESZ, (uint32_t)(n_el * ESZ), sc.bar);
    }
    // the entries past the row hold -inf (bytes the copy does not write)
    if (DT == 1) {
      for (int i = n_el + lane; i < CH; i += 32) reinterpret_cast<uint16_t*>(sc.buf)[i] = (uint16_t)Vec<DT>::NEG;
    } else {
      for (int i = n_el + lane; i < CH; i += 32) reinterpret_cast<uint32_t*>(sc.buf)[i] = Vec<DT>::NEG;
    }
    return scratch_wait(sc, p.ws.status, lane);  // (a warp-wide vote: the stores above are ordered too)
  }
  // rows off a 16-byte boundary: plain loads, -inf past the row
  if (DT == 1) {
    const uint16_t* src = static_cast<const uint16_t*>(row) + e0;
    uint16_t* dst = reinterpret_cast<uint16_t*>(sc.buf);
#pragma unroll 8
    for (int i = lane; i < CH; i += 32) dst[i] = i < n_el ? __ldcg(src + i) : (uint16_t)Vec<DT>::NEG;
  } else {
    const uint32_t* src = reinterpret_cast<const uint32_t*>(static_cast<const float*>(row) + e0);
    uint32_t* dst = reinterpret_cast<uint32_t*>(sc.buf);
#pragma unroll 8
    for (int i = lane; i < CH; i += 32) dst[i] = i < n_el ? __ldcg(src + i) : Vec<DT>::NEG;
  }
  __syncwarp();
  return true;
}

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

// Sampled chain verification of request r: rows 0..ell at slots base + k (p),
// then one draft row per set bit i of qmask (q of position i + 1).
template <int DT>
__device__ void finalize_chain_sample(const VerifyParams& p, int r, int base, int ell, uint32_t qmask, int lane,
                                      Scratch& sc) {
  if (sc.dead) return;
  constexpr int CH = Vec<DT>::CH;
  constexpr size_t ESZ = DT == 1 ? 2 : 4;
  const bool tested = lane < ell;
  const int R = ell + 1 + __popc(qmask);
  // reused draft-row partials: the drafting call recorded its log2(e) / T in
  // header word 3; another temperature is flagged (the partials stand)
  if (p.reuse_q && qmask && lane == 0 && __ldcg(p.ws.status + 3) != __float_as_uint(p.c))
    set_status(p.ws.status, SPEC_DEV_BAD_VALUE);
  const int rows_fit = min(32, VR_STAGE / (p.rowf * 8));  // rows per staging round (one copy per lane)
  const bool has_q = tested && ((qmask >> lane) & 1u);
  const int kq = has_q ? ell + 1 + __popc(qmask & ((1u << lane) - 1u)) : -1;  // lane's q row
  auto slot_of = [&](int k) -> int {
    return k <= ell ? base + k : q_slot_of(p, r, nth_bit(qmask, k - ell - 1) + 1);
  };
  // the first rows' copies go out first; the draft tokens' loads and the
  // uniforms (lane i tests position i + 1, lane ell holds the bonus's) overlap them
  stage_rows_issue(p, sc, min(R, rows_fit), slot_of, lane);
  const int yi = tested ? __ldcg(p.chain + (int64_t)r * p.L + lane) : -1;
  float u = -1.0f, u2 = 0.0f;
  if (lane <= ell) round_uniforms(p.seed, p.step, (uint32_t)r, (uint32_t)(lane + 1), &u, &u2);
  // (max, sum) of every row from its chunk partials: the rows staged a batch at
  // a time (one batch at the shapes of the configurations), G lanes per row
  float2 msp = make_float2(-INFINITY, 0.0f), msq = msp;
  float zp = 0.0f, zq = 0.0f;
  int k_lo = 0, k_hi = 0;  // the rows of the last batch
  for (int k0 = 0; k0 < R; k0 += rows_fit) {
    const int k1 = min(R, k0 + rows_fit), nr = k1 - k0;
    if (k0 > 0) stage_rows_issue(p, sc, nr, [&](int j) { return slot_of(k0 + j); }, lane);
    if (!scratch_wait(sc, p.ws.status, lane)) return;
    k_lo = k0;
    k_hi = k1;
    int G = 1;
    while (G < 32 && nr * 2 * G <= 32) G <<= 1;
    const int rr = lane / G;
    // the lane's chunks: their max first, then the rescaled sums as
    // independent terms (four accumulators), so no chain runs through the chunks
    float m = -INFINITY, s = 0.0f;
    if (rr < nr) {
      const float2* P = reinterpret_cast<const float2*>(sc.buf + (size_t)rr * p.rowf * 8);
      const int c0 = lane & (G - 1);
#pragma unroll 4
      for (int cc = c0; cc < p.nch; cc += G) m = fmaxf(m, P[cc].x);
      if (m != -INFINITY) {
        auto term = [&](int cc) -> float {  // an empty chunk (-inf, 0) weighs 0
          const float2 t = P[cc < p.nch ? cc : 0];
          const float w = t.y * ex2((t.x - m) * p.c);
          return cc < p.nch ? w : 0.0f;
        };
        float a0 = 0.0f, a1 = 0.0f, a2 = 0.0f, a3 = 0.0f;
        for (int cc = c0; cc < p.nch; cc += 4 * G) {
          a0 += term(cc);
          a1 += term(cc + G);
          a2 += term(cc + 2 * G);
          a3 += term(cc + 3 * G);
        }
        s = (a0 + a1) + (a2 + a3);
      }
    }
    for (int o = G >> 1; o >= 1; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xFFFFFFFFu, m, o), s2 = __shfl_xor_sync(0xFFFFFFFFu, s, o);
      merge_ms(m, s, m2, s2, p.c);
    }
    // lane i takes its p row (k = i) and its q row (k = kq), each merged at lane (k - k0) G;
    // a row's spare entry holds the logit at its draft token
    const bool inp = lane <= ell && lane >= k0 && lane < k1, inq = kq >= k0 && kq < k1;
    const int sp_ = inp ? (lane - k0) * G : 0, sq_ = inq ? (kq - k0) * G : 0;
    const float a0 = __shfl_sync(0xFFFFFFFFu, m, sp_), a1 = __shfl_sync(0xFFFFFFFFu, s, sp_);
    const float b0 = __shfl_sync(0xFFFFFFFFu, m, sq_), b1 = __shfl_sync(0xFFFFFFFFu, s, sq_);
    if (inp) {
      msp = make_float2(a0, a1);
      zp = reinterpret_cast<const float2*>(sc.buf + (size_t)(lane - k0) * p.rowf * 8)[p.nch].x;
    }
    if (inq) {
      msq = make_float2(b0, b1);
      zq = reinterpret_cast<const float2*>(sc.buf + (size_t)(kq - k0) * p.rowf * 8)[p.nch].x;
    }
  }
  // accept tests
  float ratio = -1.0f;
  bool acc = false;
  if (tested) {
    if (yi < 0 || yi >= p.vocab) {
      set_status(p.ws.status, SPEC_DEV_BAD_TOKEN);
      ratio = 0.0f;
    } else {
      // p(y) / q(y) = 2^((zp - mp) c) sq / (2^((zq - mq) c) sp); the quotient of
      // a fast divide (a few ulp) is far inside the 1e-5 band of the decision
      const float ep = ex2((zp - msp.x) * p.c);
      ratio = has_q ? __fdividef(ep * msq.y, ex2((zq - msq.x) * p.c) * msp.y) : __fdividef(ep, msp.y);
    }
    acc = (ratio >= 1.0f) || (u < ratio);
  }
  const unsigned fail = __ballot_sync(0xFFFFFFFFu, tested && !acc);
  const int stop = fail ? __ffs(fail) - 1 : ell;  // 0-based row that is drawn from
  if (!tested) u = -1.0f;
  const int n_acc = stop;
  for (int j = lane; j < p.L; j += 32) {
    const bool tj = j <= stop && j < ell;
    if (p.dbg_ratio) p.dbg_ratio[(int64_t)r * p.L + j] = tj ? ratio : -1.0f;
    if (p.dbg_u) p.dbg_u[(int64_t)r * p.L + j] = tj ? u : -1.0f;
  }
  for (int j = lane; j <= p.L; j += 32)
    if (j != n_acc) p.out_tokens[(int64_t)r * (p.L + 1) + j] = j < n_acc ? yi : -1;  // lane j holds y[j]
  if (lane == 0) {
    p.n_accepted[r] = n_acc;
    p.n_emitted[r] = n_acc + 1;
  }
  // the draw
  const float u2s = __shfl_sync(0xFFFFFFFFu, u2, stop);
  const float m = __shfl_sync(0xFFFFFFFFu, msp.x, stop), s = __shfl_sync(0xFFFFFFFFu, msp.y, stop);
  const bool rejected = stop < ell;
  const int y_stop = __shfl_sync(0xFFFFFFFFu, yi, stop);
  if (rejected && ((qmask >> stop) & 1u)) {
    // max(0, p - q) needs both normalisers and a second pass: resample_kernel
    const float mqs = __shfl_sync(0xFFFFFFFFu, msq.x, stop), sqs = __shfl_sync(0xFFFFFFFFu, msq.y, stop);
    if (lane == 0) {
      Record t;
      t.flag = 1;
      t.pos = stop + 1;
      t.prow = base + stop;
      t.qrow = q_slot_of(p, r, stop + 1);
      t.mp = m;
      t.sp = s;
      t.mq = mqs;
      t.sq = sqs;
      t.u2 = u2s;
      *(reinterpret_cast<Record*>(p.ws.record) + r) = t;
    }
    return;
  }
  // from p (all accepted: the bonus) or p without a rejected point mass y
  const int slot = base + stop;
  const char* row = static_cast<const char*>(p.logits) + (int64_t)slot * p.vocab * ESZ;
  const int yv = (rejected && y_stop >= 0 && y_stop < p.vocab) ? y_stop : -1;
  const int cy = yv >= 0 ? yv / CH : -1;
  const float zy = __shfl_sync(0xFFFFFFFFu, zp, stop);  // y's logit, read for its test
  const float2* P;
  if (stop >= k_lo && stop < k_hi) {
    P = reinterpret_cast<const float2*>(sc.buf + (size_t)(stop - k_lo) * p.rowf * 8);
  } else {
    if (!stage_rows(p, sc, 1, [&](int) { return slot; }, lane)) return;
    P = reinterpret_cast<const float2*>(sc.buf);
  }
  const float mc = m * p.c;
  const int per = (p.nch + 31) / 32;
  float wl[8];
  float w_cy = 0.0f;  // y's chunk without the removal
  const float w_self = yv >= 0 ? ex2(fmaf(zy, p.c, -mc)) : 0.0f;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int cc = per * lane + q;
    float w = 0.0f;
    if (q < per && cc < p.nch) {
      const float2 t = P[cc];
      w = t.y * ex2((t.x - m) * p.c);  // an empty chunk (-inf, 0) weighs 0
    }
    if (cc == cy) {
      w_cy = w;
      w = fmaxf(w - w_self, 0.0f);  // y's chunk less y's own term
    }
    wl[q] = w;
  }
  Crossing cr = find_chunk(wl, per, u2s, lane);
  int staged = -1;       // the chunk the scratch holds
  bool y_out = false;    // y's entry of the staged chunk is -inf (its bits in lane 0's y_bits)
  uint32_t y_bits = 0u;
  if (yv >= 0 && !(cr.total >= 0.0625f * s)) {
    // the residual mass is under 1/16 of the row's: y's chunk less y, summed
    // exactly instead of by the difference
    const int e0 = cy * CH, n_el = min(CH, p.vocab - e0);
    if (!stage_chunk<DT>(p, sc, row, e0, n_el, lane)) return;
    staged = cy;
    if (lane == 0) y_bits = stage_entry_swap<DT>(sc.buf, yv - e0, Vec<DT>::NEG);  // y left out
    __syncwarp();
    y_out = true;
    const float w_y = chunk_sum<DT>(sc.buf, mc, p.c, lane);
#pragma unroll
    for (int q = 0; q < 8; ++q)
      if (per * lane + q == cy) wl[q] = w_y;
    cr = find_chunk(wl, per, u2s, lane);
  }
  // the draw removes y when the residual mass exceeds 1e-30 of the row's,
  // else it falls back to p itself
  const bool remove = yv >= 0 && cr.total > 1e-30f * s;
  if (yv >= 0 && !remove) {
#pragma unroll
    for (int q = 0; q < 8; ++q)
      if (per * lane + q == cy) wl[q] = w_cy;
    cr = find_chunk(wl, per, u2s, lane);
  }
  const int e0 = cr.unit * CH, n_el = min(CH, p.vocab - e0);
  if (staged != cr.unit) {
    if (!stage_chunk<DT>(p, sc, row, e0, n_el, lane)) return;
    y_out = false;
  }
  const bool want_out = remove && cr.unit == cy;  // the draw leaves y out
  if (want_out != y_out) {
    if (lane == 0) y_bits = stage_entry_swap<DT>(sc.buf, yv - e0, want_out ? Vec<DT>::NEG : y_bits);
    __syncwarp();
  }
  float w_at;
  const int pick = chunk_draw<DT>(sc.buf, lane, cr.before, cr.t, &w_at, mc, p.c);
  if (lane == 0) {
    p.out_tokens[(int64_t)r * (p.L + 1) + n_acc] = e0 + pick;
    if (p.dbg_resid) p.dbg_resid[r] = w_at / cr.total;
  }
}

// The drafter's probabilistic token of draft row `row` (request r, position
// k + 1): y ~ softmax(z / T) by inverse CDF at word 0 of Philox counter
// (r, 0x40000000 + k + 1, lo32(step), hi32(step)), a counter domain apart from
// verification's; q(y) in dbg_resid.
template <int DT>
__device__ void finalize_draft(const VerifyParams& p, int row, int lane, Scratch& sc) {
  if (sc.dead) return;
  constexpr int CH = Vec<DT>::CH;
  constexpr size_t ESZ = DT == 1 ? 2 : 4;
  const int r = row / p.K, k = row - r * p.K;
  const int slot = q_slot_of(p, r, k + 1);
  if (!stage_rows(p, sc, 1, [&](int) { return slot; }, lane)) return;
  const float2* P = reinterpret_cast<const float2*>(sc.buf);
  const int per = (p.nch + 31) / 32;
  float lm = -INFINITY;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int cc = per * lane + q;
    if (q < per && cc < p.nch) lm = fmaxf(lm, P[cc].x);
  }
  const float m = warp_max(lm);
  uint32_t o[4];
  philox4x32_10((uint32_t)r, 0x40000000u + (uint32_t)(k + 1), (uint32_t)p.step, (uint32_t)(p.step >> 32),
                (uint32_t)p.seed, (uint32_t)(p.seed >> 32), o);
  const float u = (float)(o[0] >> 8) * (1.0f / 16777216.0f);
  int y = 0;
  float q_at = 0.0f, total = 0.0f, zy = -INFINITY;
  if (m != -INFINITY) {
    float wl[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int cc = per * lane + q;
      float w = 0.0f;
      if (q < per && cc < p.nch) {
        const float2 t = P[cc];
        w = t.y * ex2((t.x - m) * p.c);  // an empty chunk (-inf, 0) weighs 0
      }
      wl[q] = w;
    }
    const Crossing cr = find_chunk(wl, per, u, lane);
    total = cr.total;
    const int e0 = cr.unit * CH, n_el = min(CH, p.vocab - e0);
    const char* base = static_cast<const char*>(p.draft) + (int64_t)row * p.vocab * ESZ;
    if (!stage_chunk<DT>(p, sc, base, e0, n_el, lane)) return;
    const int pick = chunk_draw<DT>(sc.buf, lane, cr.before, cr.t, &q_at, m * p.c, p.c);
    y = e0 + pick;
    zy = DT == 1 ? __uint_as_float((uint32_t) reinterpret_cast<const uint16_t*>(sc.buf)[pick] << 16)
                 : reinterpret_cast<const float*>(sc.buf)[pick];
  }
  if (lane == 0) {
    // the spare entry of the row's partials: the logit at the drawn token, as
    // verification's stream would record it, so verification can reuse the
    // row's partials instead of reading the row again (and the temperature
    // they were made at)
    __stcg(&partial_row(p, slot)[p.nch], make_float2(zy, 0.0f));
    p.ws.status[3] = __float_as_uint(p.c);
    p.out_tokens[row] = y;
    if (p.dbg_u) p.dbg_u[row] = u;
    if (p.dbg_resid) p.dbg_resid[row] = total > 0.0f ? q_at / total : 0.0f;
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
  int r, item, slot, pos;  // pos: the row's 1-based position (draft rows: their position)
  const char* row;
};

// a bulk copy whose lines are marked for early eviction from L2 (the rows are
// read once; what the next kernels read stays resident)
__device__ __forceinline__ void bulk_g2s_stream(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                                uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;\n" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

template <int MODE>
__device__ __forceinline__ void locate(const VerifyParams& p, const int32_t* s_pre, const int32_t* s_base,
                                       const int32_t* s_len, const uint32_t* s_qm, int item, size_t esz,
                                       Cursor& c) {
  if (item == c.item) return;
  c.item = item;
  if constexpr (MODE == MODE_DRAFT) {  // item = draft row (request item / K, position item % K + 1)
    const int r = item / p.K, k = item - r * p.K;
    c.r = item;
    c.pos = k + 1;
    c.slot = q_slot_of(p, r, k + 1);
    c.row = static_cast<const char*>(p.draft) + (int64_t)item * p.vocab * esz;
    return;
  } else {
  while (s_pre[c.r + 1] <= item) ++c.r;
  const int li = item - s_pre[c.r];
  const int len = s_len[c.r];
  if (MODE == MODE_TREE || li <= len) {
    c.slot = s_base[c.r] + li;
    c.pos = li + 1;
    c.row = static_cast<const char*>(p.logits) + (int64_t)c.slot * p.vocab * esz;
  } else {  // the (li - len)-th position that carries a draft distribution
    const int pos = nth_bit(s_qm[c.r], li - len - 1) + 1;
    c.slot = q_slot_of(p, c.r, pos);
    c.pos = pos;
    c.row = static_cast<const char*>(p.draft) + ((int64_t)c.r * p.K + pos - 1) * p.vocab * esz;
  }
  }
}

template <int DT, int MODE>
__global__ void __launch_bounds__(VR_THREADS, 1) verify_rows_kernel(VerifyParams p) {
  constexpr size_t esz = DT == 1 ? 2 : 4;
  constexpr int CH = Vec<DT>::CH;
  constexpr bool SAMPLED = MODE == MODE_CHAIN_SAMPLE || MODE == MODE_DRAFT;
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr size_t WB = VR_WBUF(MODE);
  unsigned char* wbuf = smem + (size_t)warp * WB;  // this warp's stage (and scratch)
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)VR_WARPS * WB) + warp * VR_BARS;
  int32_t* s_pre = reinterpret_cast<int32_t*>(smem + (size_t)VR_WARPS * (WB + 8 * VR_BARS));
  int32_t* s_base = s_pre + p.batch + 1;
  int32_t* s_len = s_base + p.batch;
  uint32_t* s_qm = reinterpret_cast<uint32_t*>(s_len + p.batch);
  __shared__ int32_t s_part[VR_WARPS];

  const int B = p.batch;
  uint32_t n_items;
  if (MODE == MODE_DRAFT) {
    n_items = (uint32_t)B * (uint32_t)p.K;
  } else {
    // ---- per-request work rows (every CTA builds the same table)
    const int per_t = (B + VR_THREADS - 1) / VR_THREADS;
    int32_t my_sum = 0;
    const int32_t tot_rows = p.row_off[B];
    for (int q = 0; q < per_t; ++q) {
      const int r = tid * per_t + q;
      if (r >= B) break;
      const int32_t b0 = p.row_off[r], b1 = p.row_off[r + 1];
      const int32_t vl = MODE == MODE_TREE ? 0 : p.verify_len[r];  // issued with the offsets
      int32_t cnt = 0, len = 0;
      uint32_t qm = 0;
      bool valid;
      // the draft-distribution flags of the request's L positions, loaded
      // together with its offsets and length (they do not depend on them)
      uint32_t zf = 0;  // bit i: position i + 1 carries a draft distribution (flag 0)
      if (MODE == MODE_CHAIN_SAMPLE && p.use_q && p.pm) {
        const uint8_t* pmr = p.pm + (int64_t)r * p.L;
        uint8_t f[SPEC_MAX_L];
#pragma unroll
        for (int i = 0; i < SPEC_MAX_L; ++i) f[i] = i < p.L ? pmr[i] : (uint8_t)1;
#pragma unroll
        for (int i = 0; i < SPEC_MAX_L; ++i) zf |= (f[i] == 0 ? 1u : 0u) << i;
        asm volatile("" ::"r"(zf));  // keeps these loads beside the offsets' (not sunk past their use)
      }
      if (MODE == MODE_TREE) {
        len = b1 - b0;
        valid = b0 >= 0 && len >= 1 && len <= p.max_nodes && b1 <= tot_rows && tot_rows <= p.max_rows;
        cnt = valid ? len : 0;
      } else {
        len = vl;
        valid = len >= 0 && len <= p.L && b0 >= 0 && (int64_t)b0 + len < b1 && b1 <= tot_rows &&
                tot_rows <= p.max_rows;
        cnt = valid ? len + 1 : 0;
        if (valid && MODE == MODE_CHAIN_SAMPLE && p.use_q && p.pm) {
          // the positions that carry a draft distribution
          const uint32_t within = len >= 32 ? 0xFFFFFFFFu : (1u << len) - 1u;
          const uint32_t kmask = p.K >= 32 ? 0xFFFFFFFFu : (1u << p.K) - 1u;
          qm = zf & within & kmask;
          const bool beyond = (zf & within & ~kmask) != 0u;
          if (beyond && blockIdx.x == 0) set_status(p.ws.status, SPEC_DEV_BAD_LENGTH);
          if (!p.reuse_q) cnt += __popc(qm);  // reused draft rows are not streamed
        }
      }
      if (!valid && blockIdx.x == 0) set_status(p.ws.status, SPEC_DEV_BAD_LENGTH);
      s_base[r] = b0;
      s_len[r] = valid ? len : -1;
      s_qm[r] = qm;
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
    n_items = (uint32_t)s_pre[B];

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
  }

  // ---- this warp's contiguous range [lo, hi) of chunks (8 KB of one row each):
  // floor(gw total / nw) .. floor((gw + 1) total / nw) in 32-bit arithmetic
  // (the host bounds total below 2^31 and nw^2 below 2^31)
  const uint32_t nch = (uint32_t)p.nch;
  const uint32_t total = n_items * nch;
  const uint32_t nw = gridDim.x * VR_WARPS, gw = blockIdx.x * VR_WARPS + warp;
  const uint32_t qq = udiv(total, nw, p.m_nw), rem = total - qq * nw;
  const uint32_t lo = gw * qq + udiv(gw * rem, nw, p.m_nw), hi = (gw + 1) * qq + udiv((gw + 1) * rem, nw, p.m_nw);
  if (lo >= hi) return;
  const bool vec = p.vec_ok != 0;
  const int first = (int)udiv(lo, nch, p.m_nch);  // the item of chunk lo
  Cursor ic, cc;  // issue and consume cursors
  {
    int a = 0;
    if (MODE != MODE_DRAFT) {
      // the last r with s_pre[r] <= first (s_pre[0] = 0): the warp tests 32
      // evenly spaced candidates of [a, end) per round
      int end = B;
      while (end - a > 1) {
        const int step = (end - a + 31) >> 5;
        const int cand = a + step * lane;
        const unsigned ok = __ballot_sync(0xFFFFFFFFu, cand < end && s_pre[cand] <= first);
        a += step * (31 - __clz(ok));  // bit 0 is set: s_pre[a] <= first
        end = min(end, a + step);
      }
    }
    ic.r = cc.r = a;
    ic.item = cc.item = -1;
  }
  // the issue cursor walks (item, chunk) incrementally from lo; it locates a
  // row only when it enters it and then advances its source pointer
  int is_item = first, is_u = (int)(lo - (uint32_t)first * nch);
  const char* is_src = nullptr;
  uint64_t l2_first;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(l2_first));
  auto issue = [&](int s) {
    if (is_src == nullptr) {
      locate<MODE>(p, s_pre, s_base, s_len, s_qm, is_item, esz, ic);
      is_src = ic.row + (size_t)is_u * CH * esz;
    }
    const uint32_t bytes = (is_u + 1 < (int)nch) ? (uint32_t)VR_STAGE : (uint32_t)((p.vocab - is_u * CH) * esz);
    mbar_arrive_expect_tx(&bars[s], bytes);
    bulk_g2s_stream(wbuf + (size_t)s * VR_STAGE, is_src, bytes, &bars[s], l2_first);
    is_src += VR_STAGE;
    if (++is_u == (int)nch) {
      is_u = 0;
      ++is_item;
      is_src = nullptr;
    }
  };
  if (lane == 0) {
    for (int s = 0; s < VR_BARS; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
    if (vec)
      issue(0);
  }
  __syncwarp();

  int run_r = -1, run_slot = -1, run_y = -1;
  constexpr int s = 0;  // the stage
  uint32_t run_units = 0;
  unsigned long long run_key = 0ull;
  int bad = 0, aborted = 0;
  uint32_t w = lo;
  uint32_t ph = 0;
  Scratch sc;
  if (SAMPLED) {
    sc.buf = wbuf + VR_STAGE;
    sc.bar = &bars[1];
    sc.phase = 0;
    sc.dead = 0;
  }

  auto flush_row = [&]() {
    if ((MODE == MODE_CHAIN_GREEDY || MODE == MODE_TREE) && run_slot >= 0 && run_key != 0ull && lane == 0)
      atomicMax(&p.ws.rowkey[run_slot], run_key);
  };
  // a request's arrival: true for the warp that completes it
  auto arrive = [&]() -> bool {
    int last = 0;
    if (lane == 0) {
      // release this warp's partials / row keys, acquire everyone else's
      uint32_t* ctr = MODE == MODE_DRAFT ? &p.ws.counter3[run_r] : &p.ws.counter[run_r];
      const uint32_t need = MODE == MODE_DRAFT ? nch : (uint32_t)(s_pre[run_r + 1] - s_pre[run_r]) * nch;
      const uint32_t old = atomic_add_acq_rel(ctr, run_units);
      last = (old + run_units == need);
    }
    last = __shfl_sync(0xFFFFFFFFu, last, 0);
    if (last) __syncwarp();  // orders every lane after lane 0's acquire
    return last != 0;
  };
  auto finalize = [&](int r) {
    if (MODE == MODE_TREE)
      finalize_tree(p, r, s_base[r], s_len[r], lane);
    else if (MODE == MODE_CHAIN_GREEDY)
      finalize_chain_greedy<DT>(p, r, s_base[r], s_len[r], lane);
    else if (MODE == MODE_CHAIN_SAMPLE)
      finalize_chain_sample<DT>(p, r, s_base[r], s_len[r], s_qm[r], lane, sc);
    else
      finalize_draft<DT>(p, r, lane, sc);
    if (lane == 0) *(MODE == MODE_DRAFT ? &p.ws.counter3[r] : &p.ws.counter[r]) = 0u;
  };

  // The stream runs in an inner loop; a request this warp completes in the
  // middle of its range leaves that loop and is finalized between two chunks,
  // so the finalizer's code lies outside the loop body and the loop's own code
  // stays contiguous (a finalizer inlined inside the loop body measured as
  // instruction-cache misses on every warp of small launches).
  int item = first, u = (int)(lo - (uint32_t)first * nch);
  int pend = -1;  // a request completed by this warp, to finalize
  bool ended = false;
  while (!ended) {
  for (; w < hi; ++w) {
    locate<MODE>(p, s_pre, s_base, s_len, s_qm, item, esz, cc);
    if (cc.slot != run_slot) {
      flush_row();
      run_slot = cc.slot;
      run_key = 0ull;
      if (MODE == MODE_CHAIN_SAMPLE)  // the row's draft token (none on the bonus row)
        run_y = cc.pos <= s_len[cc.r] ? __ldcg(p.chain + (int64_t)cc.r * p.L + cc.pos - 1) : -1;
    }
    if (cc.r != run_r) {
      const bool last = run_r >= 0 && arrive();
      const int done_r = run_r;
      run_r = cc.r;
      run_units = 0;
      if (last) {
        pend = done_r;
        break;
      }
    }
    const int e0 = u * CH;
    const int n_el = min(CH, p.vocab - e0);
    const bool has_y = MODE == MODE_CHAIN_SAMPLE && run_y >= e0 && run_y < e0 + n_el;
    float zy = 0.0f;
    unsigned long long key = 0ull;
    float2 ms = make_float2(-INFINITY, 0.0f);
    if (vec) {
      const bool landed = mbar_wait_bounded(&bars[s], ph, SPEC_WAIT_POLLS);
      if (!__all_sync(0xFFFFFFFFu, landed)) {  // warp-uniform decision
        aborted = 1;
        break;
      }
      // copy the chunk to registers (and the draft token's logit) and refill
      // the stage at once, so that the next copy is in flight while the warp computes
      uint4 v[Vec<DT>::NV];
      const unsigned char* st = wbuf + (size_t)s * VR_STAGE;
      vec_load_smem<DT>(st, n_el, lane, v);
      if (has_y)
        zy = DT == 1 ? __uint_as_float((uint32_t) reinterpret_cast<const uint16_t*>(st)[run_y - e0] << 16)
                     : reinterpret_cast<const float*>(st)[run_y - e0];
      __syncwarp();
      if (lane == 0 && w + 1 < hi) issue(s);
      if (SAMPLED)
        ms = unit_softmax_vec<DT, 0, Vec<DT>::NV>(v, p.c, bad);
      else if (DT == 1)
        key = chunk_argmax_bf16(v, n_el, lane, bad);
      else
        key = unit_argmax_vec<DT>(v, n_el, lane, bad);
    } else {
      if (has_y) zy = load_one<DT>(cc.row, run_y);
#pragma unroll
      for (int j = 0; j < Vec<DT>::SUB; ++j) {
        const int e1 = e0 + j * SPEC_UNIT;
        const int n1 = min(SPEC_UNIT, p.vocab - e1);
        if (n1 <= 0) continue;
        const void* unit = cc.row + (size_t)e1 * esz;
        if (SAMPLED) {
          const float2 t = unit_softmax_scalar<DT>(unit, n1, lane, p.c, bad);
          merge_ms(ms.x, ms.y, t.x, t.y, p.c);
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
    if (SAMPLED) {
      if (lane == 0) {
        float2* pr = partial_row(p, cc.slot);
        __stcg(&pr[u], ms);
        if (has_y) __stcg(&pr[p.nch], make_float2(zy, 0.0f));
      }
    } else if (key != 0ull) {
      // rebase the chunk offset to the row index; keys of one row fold by max
      const int32_t idx = argmax_key_index(key) + e0;
      const unsigned long long kk =
          (key & 0xFFFFFFFF00000000ull) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)idx);
      if (kk > run_key) run_key = kk;
    }
    ++run_units;
    if (++u == (int)nch) {
      u = 0;
      ++item;
    }
    ph ^= 1u;
  }
  if (aborted) break;
  if (pend < 0) {  // the range is done: the last request's arrival
    flush_row();
    if (run_r >= 0 && arrive()) pend = run_r;
    ended = true;
  }
  if (pend >= 0) {
    finalize(pend);
    pend = -1;
  }
  }
  if (aborted) {
    // a copy did not land in time: record it, wait (bounded) once more for
    // the copy this warp has in flight, and stop without finalizing
    if (lane == 0) {
      set_status(p.ws.status, SPEC_DEV_TIMEOUT);
      mbar_wait_bounded(&bars[0], ph, SPEC_WAIT_POLLS);
    }
    __syncwarp();
    return;
  }
  if (SAMPLED && sc.dead && lane == 0) mbar_wait_bounded(sc.bar, sc.phase ^ 1u, SPEC_WAIT_POLLS);  // the copy given up on
  if (bad && lane == 0) set_status(p.ws.status, SPEC_DEV_NONFINITE);
}

// ------------------------------------------------------------------ draw from max(0, p - q)
// N consecutive entries of a row from entry e (fp32; -inf past the row's end)
template <int DT, int N>
__device__ __forceinline__ void load_entries(const void* row, int e, int vocab, bool vec, float (&x)[N]) {
  if (vec) {
    constexpr int PV = DT == 1 ? 8 : 4;  // entries per 16-byte vector
    uint4 w[N / PV];
#pragma unroll
    for (int k = 0; k < N / PV; ++k)
      w[k] = e + PV * k < vocab ? __ldcg(reinterpret_cast<const uint4*>(static_cast<const char*>(row) +
                                                                         (size_t)(e + PV * k) * (DT == 1 ? 2 : 4)))
                                : make_uint4(Vec<DT>::NEG, Vec<DT>::NEG, Vec<DT>::NEG, Vec<DT>::NEG);
#pragma unroll
    for (int k = 0; k < N / PV; ++k) {
      const uint32_t q4[4] = {w[k].x, w[k].y, w[k].z, w[k].w};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        if (DT == 1) {
          x[PV * k + 2 * h] = bf16_lo(q4[h]);
          x[PV * k + 2 * h + 1] = bf16_hi(q4[h]);
        } else {
          x[PV * k + h] = __uint_as_float(q4[h]);
        }
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < N; ++j) x[j] = e + j < vocab ? load_one<DT>(row, e + j) : -INFINITY;
  }
}

// One CTA per (chunk c, request r) with a record: the chunk's mass of
// max(0, p - q) at the rejected position (warp sums, then one exchange); the
// last CTA of the request (arrival counter) draws: warp 0 locates the crossing
// chunk over the chunks' masses at u' of their total (p itself when that mass
// is at most 1e-30), then every thread takes PER consecutive entries of that
// chunk, and the one thread whose running range holds the crossing (or, when
// rounding leaves none, holds the last entry with mass) walks its entries and
// writes the token.  Every step but the walk is warp-wide: six CTA barriers.
template <int DT>
__global__ void __launch_bounds__(RS_THREADS) resample_kernel(VerifyParams p) {
  constexpr int CH = Vec<DT>::CH, PER = CH / RS_THREADS;  // 16 bf16 / 8 fp32 entries per thread
  constexpr int NW = RS_THREADS / 32;
  constexpr size_t ESZ = DT == 1 ? 2 : 4;
  __shared__ __align__(16) Record s_rec;
  __shared__ float s_w[NW];
  __shared__ int s_last, s_cx;
  __shared__ float s_t[3];  // the crossing chunk's weight before it (-1: last mode), the total, t
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int c = blockIdx.x, r = blockIdx.y;
  if (tid < 4)
    reinterpret_cast<uint4*>(&s_rec)[tid] =
        __ldcg(reinterpret_cast<const uint4*>(reinterpret_cast<const Record*>(p.ws.record) + r) + tid);
  __syncthreads();
  if (!s_rec.flag) return;
  const Record rec = s_rec;
  const bool vec = p.vec_ok != 0;
  const char* prow = static_cast<const char*>(p.logits) + (int64_t)rec.prow * p.vocab * ESZ;
  const char* qrow = static_cast<const char*>(p.draft) + ((int64_t)r * p.K + rec.pos - 1) * p.vocab * ESZ;
  const float ip = 1.0f / rec.sp, iq = 1.0f / rec.sq;
  const float mpc = rec.mp * p.c, mqc = rec.mq * p.c;
  // weights of logits (2^-inf = +0 covers the empty entries)
  auto pw = [&](float z) -> float { return ex2(fmaf(z, p.c, -mpc)) * ip; };
  auto resid = [&](float zp, float zq) -> float {
    const float a = pw(zp);
    const float b = ex2(fmaf(zq, p.c, -mqc)) * iq;
    return fmaxf(a - b, 0.0f);
  };
  float* masses = reinterpret_cast<float*>(p.ws.partial2) + (int64_t)r * p.pstride;
  {
    float zp[PER], zq[PER];
    load_entries<DT, PER>(prow, c * CH + PER * tid, p.vocab, vec, zp);
    load_entries<DT, PER>(qrow, c * CH + PER * tid, p.vocab, vec, zq);
    float sum = 0.0f;
#pragma unroll
    for (int j = 0; j < PER; ++j) sum += resid(zp[j], zq[j]);
    sum = warp_sum(sum);
    if (lane == 0) s_w[warp] = sum;
    __syncthreads();
    if (tid == 0) {
      float tot = 0.0f;
#pragma unroll
      for (int q = 0; q < NW; ++q) tot += s_w[q];
      __stcg(&masses[c], tot);
      // release this chunk's mass, acquire the others'
      s_last = atomic_add_acq_rel(&p.ws.counter2[r], 1u) + 1u == (uint32_t)p.nch;
    }
    __syncthreads();
    if (!s_last) return;
  }
  // ---- the last CTA of request r draws.  Warp 0: the crossing chunk over the
  // masses (8 per lane at most; p's chunk weights when the residual is empty)
  if (warp == 0) {
    const int per = (p.nch + 31) / 32;
    float wl[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int cc = per * lane + q;
      wl[q] = (q < per && cc < p.nch) ? __ldcg(&masses[cc]) : 0.0f;
    }
    Crossing cr = find_chunk(wl, per, rec.u2, lane);
    const int fallback = !(cr.total > 1e-30f);
    if (fallback) {  // no residual mass: the draw falls back to p
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int cc = per * lane + q;
        float w = 0.0f;
        if (q < per && cc < p.nch) {
          const float2 t = __ldcg(&partial_row(p, rec.prow)[cc]);
          w = t.y * ex2((t.x - rec.mp) * p.c) * ip;
        }
        wl[q] = w;
      }
      cr = find_chunk(wl, per, rec.u2, lane);
    }
    if (lane == 0) {
      s_cx = cr.unit | (fallback << 30);
      s_t[0] = cr.before;
      s_t[1] = cr.total;
      s_t[2] = cr.t;
    }
  }
  __syncthreads();
  const int cx = s_cx & 0x3FFFFFFF;
  const bool fallback = (s_cx >> 30) != 0;
  const float before = s_t[0], total = s_t[1];
  const bool last_mode = before < 0.0f;  // t at or above the total: the last entry with mass
  const float tt = last_mode ? INFINITY : s_t[2] - before;
  // ---- the crossing chunk's entries, PER consecutive ones per thread
  float wv[PER], sum = 0.0f;
  {
    float zp[PER], zq[PER];
    load_entries<DT, PER>(prow, cx * CH + PER * tid, p.vocab, vec, zp);
    if (!fallback) load_entries<DT, PER>(qrow, cx * CH + PER * tid, p.vocab, vec, zq);
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      wv[j] = fallback ? pw(zp[j]) : resid(zp[j], zq[j]);
      sum += wv[j];
    }
  }
  // this thread's running weight over the chunk, in thread order: excl is
  // the previous thread's incl bit for bit (a shuffle within the warp, the same
  // sums across warps), so the ranges [excl, incl) tile [0, ctot) exactly
  const float winc = warp_incl_scan(sum);
  const float wprev = __shfl_up_sync(0xFFFFFFFFu, winc, 1);
  if (lane == 31) s_w[warp] = winc;
  if (tid == 0) s_last = -1;  // (read again below as the writer's key)
  __syncthreads();
  float wbefore = 0.0f, ctot = 0.0f;
#pragma unroll
  for (int q = 0; q < NW; ++q) {
    const float t = s_w[q];
    if (q < warp) wbefore += t;
    ctot += t;
  }
  const float incl = wbefore + winc, excl = lane == 0 ? wbefore : wbefore + wprev;
  // the writer: the thread whose range holds the crossing (one at most), else
  // the last thread with mass; a key picks exactly one (rounding could leave
  // several threads at the total)
  const float tc = fmaxf(tt, 0.0f);
  const bool cross = !last_mode && sum > 0.0f && excl <= tc && tc < incl;
  const bool lastpos = sum > 0.0f && incl == ctot && (last_mode || !(tc < ctot));
  if (cross || lastpos) atomicMax(&s_last, cross ? RS_THREADS + tid : tid);
  __syncthreads();
  const int key = s_last;
  if (key >= 0 && tid == (key & (RS_THREADS - 1))) {
    int pick = -1, lp = -1;
    float wp = 0.0f, lw = 0.0f, run = excl;
#pragma unroll
    for (int j = 0; j < PER; ++j)
      if (wv[j] > 0.0f) {
        run += wv[j];
        if (pick < 0 && key >= RS_THREADS && run > tc) {
          pick = j;
          wp = wv[j];
        }
        lp = j;
        lw = wv[j];
      }
    if (pick < 0) {  // rounding inside the thread, or the last entry with mass
      pick = lp;
      wp = lw;
    }
    p.out_tokens[(int64_t)r * (p.L + 1) + rec.pos - 1] = cx * CH + PER * tid + pick;
    if (p.dbg_resid) p.dbg_resid[r] = wp / total;
  } else if (key < 0 && tid == 0) {  // no entry of the chunk has mass (not reached in exact arithmetic)
    p.out_tokens[(int64_t)r * (p.L + 1) + rec.pos - 1] = cx * CH;
    if (p.dbg_resid) p.dbg_resid[r] = 0.0f;
  }
  if (tid == 0) {
    reinterpret_cast<Record*>(p.ws.record)[r].flag = 0;
    p.ws.counter2[r] = 0u;
  }
}

}  // namespace spec

// ---------------------------------------------------------------------------
// host launchers (called from api.cu)
// ---------------------------------------------------------------------------
namespace {

template <int DT, int MODE>
cudaError_t launch_rows(const spec::VerifyParams& p0, int num_sms, cudaStream_t stream) {
  spec::VerifyParams p = p0;
  p.m_nw = ((uint64_t)1 << 32) / (uint64_t)(num_sms * VR_WARPS) + 1;
  p.m_nch = ((uint64_t)1 << 32) / (uint64_t)p.nch + 1;
  const size_t table = MODE == spec::MODE_DRAFT ? 0 : (size_t)(4 * p.batch + 1) * sizeof(int32_t);
  const size_t smem = (size_t)VR_WARPS * (VR_WBUF(MODE) + 8 * VR_BARS) + table;
  auto k = spec::verify_rows_kernel<DT, MODE>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  // one CTA per SM: the shared-memory stages hold the bytes in flight
  k<<<num_sms, VR_THREADS, smem, stream>>>(p);
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
  v.partial2 = reinterpret_cast<float*>(b + ws->off_partial2);
  v.units = ws->units;
  v.max_rows = ws->max_rows;
  v.max_batch = ws->max_batch;
  v.K = ws->K;
  return v;
}

// the chunk geometry of a call: chunks per row, the staged partial row and the
// workspace's partial row stride
void set_chunks(spec::VerifyParams& p, int dtype, const spec_workspace* ws) {
  const int ch = dtype == SPEC_BF16 ? spec::Vec<1>::CH : spec::Vec<0>::CH;
  p.nch = (p.vocab + ch - 1) / ch;
  p.rowf = (p.nch + 2) & ~1;
  // the call's rows lie rowf apart (<= the workspace's stride for the finest
  // chunking), so consecutive slots are one contiguous block
  p.pstride = p.rowf;
  (void)ws;
}

}  // namespace

// The largest vocabulary (a row's chunk weights fit 8 per lane, and the draw
// kernel gives each chunk one thread) and the bound on a launch's chunks
// (32-bit work split).
extern "C" int spec_verify_limits_ok(int32_t vocab, int32_t dtype, int64_t rows, int num_sms) {
  const int ch = dtype == SPEC_BF16 ? spec::Vec<1>::CH : spec::Vec<0>::CH;
  const int64_t nch = ((int64_t)vocab + ch - 1) / ch;
  const int64_t nw = (int64_t)num_sms * VR_WARPS;
  return vocab <= SPEC_MAX_VOCAB && rows * nch < ((int64_t)1 << 31) && nw * nw < ((int64_t)1 << 31);
}

extern "C" cudaError_t spec_launch_verify_chain(
    int32_t batch, int32_t vocab, int32_t dtype, const void* logits, const int32_t* row_off,
    const void* draft, int32_t K, const int32_t* chain, int32_t L, const int32_t* verify_len,
    const uint8_t* pm, float temperature, uint64_t seed, uint64_t step, int32_t* out_tokens,
    int32_t* n_accepted, int32_t* n_emitted, float* dbg_ratio, float* dbg_u, float* dbg_resid,
    int32_t q_reuse_base, const spec_workspace* ws, int num_sms, cudaStream_t stream) {
  spec::VerifyParams p = {};
  p.batch = batch;
  p.vocab = vocab;
  p.logits = logits;
  p.row_off = row_off;
  p.max_rows = ws->max_rows;
  p.qbase = ws->max_rows;
  p.draft = draft;
  p.K = draft ? K : 0;
  p.chain = chain;
  p.L = L;
  p.verify_len = verify_len;
  p.pm = pm;
  const bool greedy = !(temperature > 0.0f);
  p.use_q = (!greedy && draft != nullptr && pm != nullptr) ? 1 : 0;
  // reused draft rows: their partials where the drafting call wrote them
  p.reuse_q = p.use_q && q_reuse_base >= 0 ? 1 : 0;
  if (p.reuse_q) p.qbase = q_reuse_base;
  p.c = greedy ? 0.0f : (float)(1.4426950408889634 / (double)temperature);
  p.seed = seed;
  p.step = step;
  p.out_tokens = out_tokens;
  p.n_accepted = n_accepted;
  p.n_emitted = n_emitted;
  p.dbg_ratio = dbg_ratio;
  p.dbg_u = dbg_u;
  p.dbg_resid = dbg_resid;
  set_chunks(p, dtype, ws);
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
  const dim3 grid((unsigned)p.nch, (unsigned)batch);
  if (dtype == SPEC_BF16)
    spec::resample_kernel<1><<<grid, RS_THREADS, 0, stream>>>(p);
  else
    spec::resample_kernel<0><<<grid, RS_THREADS, 0, stream>>>(p);
  return cudaGetLastError();
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
  p.qbase = ws->max_rows;
  p.tok = tok;
  p.parent = parent;
  p.max_nodes = max_nodes;
  p.path = path;
  p.accept_len = accept_len;
  p.out_tokens = out_tokens;
  set_chunks(p, dtype, ws);
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
  p.qbase = ws->max_rows;
  p.draft = draft_logits;
  p.K = K;
  p.c = (float)(1.4426950408889634 / (double)temperature);
  p.seed = seed;
  p.step = step;
  p.out_tokens = y;
  p.dbg_u = dbg_u;
  p.dbg_resid = dbg_q;
  set_chunks(p, dtype, ws);
  const size_t esz = dtype == SPEC_BF16 ? 2 : 4;
  p.vec_ok = (((size_t)vocab * esz) % 16 == 0 && (reinterpret_cast<uintptr_t>(draft_logits) & 15u) == 0) ? 1 : 0;
  p.ws = ws_view(ws);
  if (batch == 0) return cudaSuccess;
  return dtype == SPEC_BF16 ? launch_rows<1, spec::MODE_DRAFT>(p, num_sms, stream)
                            : launch_rows<0, spec::MODE_DRAFT>(p, num_sms, stream);
}
