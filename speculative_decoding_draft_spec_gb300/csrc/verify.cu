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
// GB300 layout.  The HBM-bound part is one pass over every verify row.  A
// persistent grid (SMs x resident CTAs) hands out work items of one warp =
// one 2048-entry unit of one row, in row-major order, so every warp streams a
// contiguous 4 KB (bf16) / 8 KB (fp32) block with 16-byte non-allocating
// loads, all issued before use.  Per unit a warp produces
//   greedy rows:  a packed 64-bit (ordered value, ~index) key, folded into the
//                 row's key with one atomicMax (largest value, lowest index);
//   sampled rows: (max, sum of 2^((z - max) log2e / T)) in the workspace.
// Each request has an arrival counter; the warp that completes a request's
// last unit (threadfence + atomicAdd, no waiting) finalizes it: argmax
// compare or Philox accept tests, and for a draw the inverse CDF in
// vocabulary order located first over the units' sums and then inside the
// one unit that holds the crossing (a second read of 4-8 KB, not of the row).
// A draw from max(0, p - q) needs both normalisers first; those requests are
// finished by a second, small kernel over the rejected (p, q) row pairs.
#include <cuda_bf16.h>

#include "common.cuh"

namespace spec {

enum { MODE_CHAIN_GREEDY = 0, MODE_CHAIN_SAMPLE = 1, MODE_TREE = 2 };
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
// greedy: fold the unit's (max, lowest index) into the row key
template <int DT>
__device__ __forceinline__ void unit_argmax(const VerifyParams& p, const void* row, int u, int slot,
                                            int lane) {
  const int e0 = u * SPEC_UNIT;
  const int n_el = min(SPEC_UNIT, p.vocab - e0);
  const bool vec = p.vec_ok != 0;
  int bad = 0;
  float lane_max = -INFINITY;
  int idx = 0x7FFFFFFF;
  float wm;
  if (DT == 1 && vec) {
    // bf16 pairs: packed max on the tensor-free HMNMX2 path, NaN pairs ignored
    const uint16_t* rp = static_cast<const uint16_t*>(row) + e0;
    uint4 w[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int vv = lane + 32 * k;
      w[k] = (8 * vv < n_el) ? ldg_stream(rp + 8 * vv)
                             : make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
    }
    __nv_bfloat162 m2 = __floats2bfloat162_rn(-INFINITY, -INFINITY);
    uint32_t nan = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint32_t ws[4] = {w[k].x, w[k].y, w[k].z, w[k].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t word = ws[q];
        m2 = __hmax2(m2, *reinterpret_cast<const __nv_bfloat162*>(&word));
        nan |= __vcmpgtu2(word & 0x7FFF7FFFu, 0x7F807F80u);
      }
    }
    bad = nan != 0;
    lane_max = fmaxf(__low2float(m2), __high2float(m2));
    wm = warp_max(lane_max);
    if (lane_max == wm) {
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int vv = lane + 32 * k;
        const uint32_t ws[4] = {w[k].x, w[k].y, w[k].z, w[k].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (idx == 0x7FFFFFFF && 8 * vv < n_el) {
            if (bf16_lo(ws[q]) == wm)
              idx = 8 * vv + 2 * q;
            else if (bf16_hi(ws[q]) == wm)
              idx = 8 * vv + 2 * q + 1;
          }
        }
      }
    }
  } else {
    float v[64];
    load_unit<DT>(row, e0, n_el, vec, lane, v);
#pragma unroll
    for (int j = 0; j < 64; ++j) {
      lane_max = fmaxf(lane_max, v[j]);
      bad |= (v[j] != v[j]);
    }
    wm = warp_max(lane_max);
    if (lane_max == wm) {
#pragma unroll
      for (int j = 0; j < 64; ++j) {
        const int i = idx_strided<DT>(lane, j, vec);
        if (i < n_el && v[j] == wm && i < idx) idx = i;
      }
    }
  }
  if (wm == INFINITY) bad = 1;
  // lowest index among the lanes holding the maximum
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) idx = min(idx, __shfl_xor_sync(0xFFFFFFFFu, idx, o));
  if (__any_sync(0xFFFFFFFFu, bad) && lane == 0) set_status(p.ws.status, SPEC_DEV_NONFINITE);
  if (lane == 0 && idx != 0x7FFFFFFF) atomicMax(&p.ws.rowkey[slot], argmax_key(wm, e0 + idx));
}

// sampled: (max, sum 2^((z - max) c)) of the unit
template <int DT>
__device__ __forceinline__ void unit_softmax(const VerifyParams& p, const void* row, int u, int slot,
                                             int lane) {
  const int e0 = u * SPEC_UNIT;
  const int n_el = min(SPEC_UNIT, p.vocab - e0);
  float v[64];
  load_unit<DT>(row, e0, n_el, p.vec_ok != 0, lane, v);
  float lm = -INFINITY;
#pragma unroll
  for (int j = 0; j < 64; ++j) lm = fmaxf(lm, v[j]);
  const float m = warp_max(lm);
  float s = 0.0f;
  if (m != -INFINITY) {
    const float mc = m * p.c;
#pragma unroll
    for (int j = 0; j < 64; ++j) s += ex2(fmaf(v[j], p.c, -mc));
  }
  s = warp_sum(s);
  if (lane == 0) {
    if (!(s == s) || m == INFINITY) set_status(p.ws.status, SPEC_DEV_NONFINITE);
    __stcg(&p.ws.partial[(int64_t)slot * p.ws.units + u], make_float2(m, s));
  }
}

// ------------------------------------------------------------------ helpers
// (max, sum) of a whole row from its unit partials; every lane gets the result
__device__ __forceinline__ float2 merge_row(const VerifyParams& p, int slot, int lane) {
  float m = -INFINITY, s = 0.0f;
  for (int u = lane; u < p.units; u += 32) {
    const float2 t = __ldcg(&p.ws.partial[(int64_t)slot * p.ws.units + u]);
    if (t.x == -INFINITY) continue;
    if (t.x > m) {
      s = s * ex2((m - t.x) * p.c) + t.y;
      m = t.x;
    } else {
      s += t.y * ex2((t.x - m) * p.c);
    }
  }
  const float M = warp_max(m);
  const float sc = (m == -INFINITY) ? 0.0f : s * ex2((m - M) * p.c);
  return make_float2(M, warp_sum(sc));
}

// Inverse CDF over unit weights w_u (unit order) held as 3+ consecutive units
// per lane: returns the unit holding the crossing of t and the weight before it.
// units_per_lane consecutive units belong to each lane, so lane order is unit order.
struct Crossing {
  int unit;
  double before;
  double total;
};

template <typename WFn>
__device__ __forceinline__ Crossing find_unit(int units, double t, int lane, WFn wfn) {
  const int per = (units + 31) / 32;
  const int u0 = lane * per;
  double lsum = 0.0;
  int last_pos = -1;
  for (int q = 0; q < per; ++q) {
    const int u = u0 + q;
    if (u < units) {
      const double w = wfn(u);
      lsum += w;
      if (w > 0.0) last_pos = u;
    }
  }
  const double incl = warp_incl_scan_d(lsum);
  const double excl = incl - lsum;
  const double total = __shfl_sync(0xFFFFFFFFu, incl, 31);
  const unsigned hit = __ballot_sync(0xFFFFFFFFu, incl > t && lsum > 0.0);
  Crossing c;
  c.total = total;
  if (hit) {
    const int src = __ffs(hit) - 1;
    int unit = -1;
    double before = 0.0;
    if (lane == src) {
      double run = excl;
      for (int q = 0; q < per; ++q) {
        const int u = u0 + q;
        if (u >= units) break;
        const double w = wfn(u);
        if (run + w > t && w > 0.0) {
          unit = u;
          before = run;
          break;
        }
        run += w;
      }
      if (unit < 0) {  // rounding inside the lane: its last unit with mass
        unit = last_pos;
        before = incl - (last_pos >= 0 ? wfn(last_pos) : 0.0);
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
    c.before = -1.0;  // marker: take the last positive entry of the unit
  }
  return c;
}

// inside one unit: the smallest index whose running sum (from `before`)
// exceeds t, over residual values r[64] in contiguous lane layout.  Returns
// (index within the unit, r at that index); falls back to the last positive.
__device__ __forceinline__ int find_in_unit(const float r[64], double before, double t, int lane,
                                            float* r_at) {
  double lsum = 0.0;
#pragma unroll
  for (int j = 0; j < 64; ++j) lsum += (double)r[j];
  const double incl = warp_incl_scan_d(lsum) + (before < 0.0 ? 0.0 : before);
  const double excl = incl - lsum;
  int pick = -1;
  float rv = 0.0f;
  const bool last_mode = before < 0.0;
  const unsigned hit = last_mode ? 0u : __ballot_sync(0xFFFFFFFFu, incl > t && lsum > 0.0);
  if (hit) {
    const int src = __ffs(hit) - 1;
    if (lane == src) {
      double run = excl;
      int lastp = -1;
      for (int j = 0; j < 64; ++j) {
        if (r[j] > 0.0f) lastp = j;
        run += (double)r[j];
        if (run > t && r[j] > 0.0f) {
          pick = 64 * lane + j;
          rv = r[j];
          break;
        }
      }
      if (pick < 0 && lastp >= 0) {
        pick = 64 * lane + lastp;
        rv = r[lastp];
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
  int a = 0;
  if (lane <= ell) {
    unsigned long long* kp = &p.ws.rowkey[base + lane];
    const unsigned long long key = __ldcg(kp);
    a = key ? argmax_key_index(key) : 0;  // an all-NaN row: 0 (flagged already)
    *kp = 0ull;
  }
  const int yi = lane < ell ? y[lane] : -1;
  const bool tested = lane < ell;
  if (tested && (yi < 0 || yi >= p.vocab)) set_status(p.ws.status, SPEC_DEV_BAD_TOKEN);
  const bool ok = tested && yi == a;
  const unsigned fail = __ballot_sync(0xFFFFFFFFu, tested && !ok);
  const int stop = fail ? __ffs(fail) - 1 : ell;  // 0-based row of the emitted argmax
  const int n_acc = stop;
  const int a_stop = __shfl_sync(0xFFFFFFFFu, a, stop);
  for (int j = lane; j <= p.L; j += 32) {
    int t = -1;
    if (j < n_acc) t = y[j];
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
  // (max, sum) of each p row (lane i keeps row i) and each q row (lane i-1)
  float mrow = 0.0f, srow = 0.0f, mq = 0.0f, sq = 0.0f;
  int use_q_lane = 0;
  for (int i = 0; i <= ell; ++i) {
    const float2 ms = merge_row(p, base + i, lane);
    if (lane == i) {
      mrow = ms.x;
      srow = ms.y;
    }
  }
  for (int i = 1; i <= ell; ++i) {
    const int uq = p.use_q && pmr && pmr[i - 1] == 0 && i <= p.K;
    if (uq) {
      const float2 ms = merge_row(p, q_slot_of(p, r, i), lane);
      if (lane == i - 1) {
        mq = ms.x;
        sq = ms.y;
        use_q_lane = 1;
      }
    }
  }
  // accept tests: lane i-1 tests position i
  const bool tested = lane < ell;
  float ratio = -1.0f, u = -1.0f, u2 = 0.0f;
  bool acc = false;
  int yi = -1;
  if (tested) {
    yi = y[lane];
    round_uniforms(p.seed, p.step, (uint32_t)r, (uint32_t)(lane + 1), &u, &u2);
    if (yi < 0 || yi >= p.vocab) {
      set_status(p.ws.status, SPEC_DEV_BAD_TOKEN);
      ratio = 0.0f;
    } else {
      const float zp = load_one<DT>(p.logits, (int64_t)(base + lane) * p.vocab + yi);
      const float py = ex2((zp - mrow) * p.c) / srow;
      if (use_q_lane) {
        const float zq = load_one<DT>(p.draft, ((int64_t)r * p.K + lane) * p.vocab + yi);
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
    if (j != n_acc) p.out_tokens[(int64_t)r * (p.L + 1) + j] = j < n_acc ? y[j] : -1;
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
  // weight of the unit holding y with y removed: a rescan of that one unit
  double w_y = 0.0;
  if (u_y >= 0) {
    float v[64];
    const int e0 = u_y * SPEC_UNIT;
    const int n_el = min(SPEC_UNIT, p.vocab - e0);
    load_unit_contig<DT>(row, e0, n_el, vec, lane, v);
    const float mc = m * p.c;
    double ls = 0.0;
#pragma unroll
    for (int j = 0; j < 64; ++j)
      if (e0 + 64 * lane + j != yv && v[j] != -INFINITY) ls += (double)ex2(fmaf(v[j], p.c, -mc));
    w_y = warp_sum_d(ls);
  }
  auto w_plain = [&](int uu) -> double {
    const float2 t = __ldcg(&p.ws.partial[(int64_t)slot * p.ws.units + uu]);
    if (t.x == -INFINITY) return 0.0;
    return (double)(t.y * ex2((t.x - m) * p.c));
  };
  auto w_removed = [&](int uu) -> double { return uu == u_y ? w_y : w_plain(uu); };
  // residual mass (unnormalised); a residual at or below 1e-30 of the row's
  // mass falls back to p itself
  bool remove = false;
  double total;
  if (yv >= 0) {
    double ls = 0.0;
    for (int uu = lane; uu < p.units; uu += 32) ls += w_removed(uu);
    total = warp_sum_d(ls);
    remove = total > 1e-30 * (double)s;
  }
  if (!remove) {
    double ls = 0.0;
    for (int uu = lane; uu < p.units; uu += 32) ls += w_plain(uu);
    total = warp_sum_d(ls);
  }
  const double t = (double)u2_stop * total;
  const Crossing cr = remove ? find_unit(p.units, t, lane, w_removed) : find_unit(p.units, t, lane, w_plain);
  float v[64];
  const int e0 = cr.unit * SPEC_UNIT;
  const int n_el = min(SPEC_UNIT, p.vocab - e0);
  load_unit_contig<DT>(row, e0, n_el, vec, lane, v);
  const float mc = m * p.c;
#pragma unroll
  for (int j = 0; j < 64; ++j) {
    const int gi = e0 + 64 * lane + j;
    v[j] = ((remove && gi == yv) || v[j] == -INFINITY) ? 0.0f : ex2(fmaf(v[j], p.c, -mc));
  }
  float r_at;
  const int pick = find_in_unit(v, cr.before, t, lane, &r_at);
  if (lane == 0) {
    p.out_tokens[(int64_t)r * (p.L + 1) + n_acc] = e0 + pick;
    if (p.dbg_resid) p.dbg_resid[r] = (float)((double)r_at / total);
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
template <int DT, int MODE>
__global__ void __launch_bounds__(SPEC_CTA_THREADS, 2) verify_rows_kernel(VerifyParams p) {
  extern __shared__ __align__(16) int32_t sm[];
  int32_t* s_pre = sm;                   // [batch + 1] exclusive prefix of work rows
  int32_t* s_base = sm + p.batch + 1;    // [batch] first row
  int32_t* s_len = s_base + p.batch;     // [batch] verify_len (chain) or nodes (tree)
  __shared__ int32_t s_part[SPEC_CTA_THREADS];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int B = p.batch;
  // ---- per-request row counts (every CTA computes the same table)
  const int per_t = (B + SPEC_CTA_THREADS - 1) / SPEC_CTA_THREADS;
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
    s_pre[r] = cnt;  // counts for now
    my_sum += cnt;
  }
  // block exclusive scan of the per-thread sums, then each thread's range
  s_part[tid] = my_sum;
  __syncthreads();
  for (int o = 1; o < SPEC_CTA_THREADS; o <<= 1) {
    const int32_t t = tid >= o ? s_part[tid - o] : 0;
    __syncthreads();
    s_part[tid] += t;
    __syncthreads();
  }
  {
    int32_t run = s_part[tid] - my_sum;
    for (int q = 0; q < per_t; ++q) {
      const int r = tid * per_t + q;
      if (r >= B) break;
      const int32_t cnt = s_pre[r];
      s_pre[r] = run;
      run += cnt;
    }
    if (tid == SPEC_CTA_THREADS - 1) s_pre[B] = s_part[tid];
  }
  __syncthreads();

  // ---- outputs of invalid requests (CTA 0 only)
  if (blockIdx.x == 0) {
    for (int r = warp; r < B; r += SPEC_WARPS_PER_CTA) {
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

  // ---- stream the units
  const int units = p.units;
  const int64_t total = (int64_t)s_pre[B] * units;
  const int64_t nwarps = (int64_t)gridDim.x * SPEC_WARPS_PER_CTA;
  for (int64_t w = (int64_t)blockIdx.x * SPEC_WARPS_PER_CTA + warp; w < total; w += nwarps) {
    const int32_t item = (int32_t)(w / units);
    const int u = (int)(w - (int64_t)item * units);
    // request owning this row: the last r with s_pre[r] <= item
    int lo = 0, hi = B - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_pre[mid] <= item)
        lo = mid;
      else
        hi = mid - 1;
    }
    const int r = lo;
    const int li = item - s_pre[r];
    const int len = s_len[r];
    int slot;
    const void* row;
    const size_t esz = DT == 1 ? 2 : 4;
    if (MODE == MODE_TREE || li <= len) {
      slot = s_base[r] + li;
      row = static_cast<const char*>(p.logits) + (int64_t)slot * p.vocab * esz;
    } else {
      // the (li - len)-th position (1-based) that carries a draft distribution
      int want = li - len, pos = 0;
      const uint8_t* pmr = p.pm + (int64_t)r * p.L;
      for (int i = 1; i <= len && i <= p.K; ++i)
        if (pmr[i - 1] == 0 && --want == 0) {
          pos = i;
          break;
        }
      slot = q_slot_of(p, r, pos);
      row = static_cast<const char*>(p.draft) + ((int64_t)r * p.K + pos - 1) * p.vocab * esz;
    }
    if (MODE == MODE_CHAIN_SAMPLE)
      unit_softmax<DT>(p, row, u, slot, lane);
    else
      unit_argmax<DT>(p, row, u, slot, lane);

    // arrival: the warp that completes the request finalizes it
    int last = 0;
    if (lane == 0) {
      __threadfence();
      const uint32_t need = (uint32_t)((s_pre[r + 1] - s_pre[r]) * units);
      const uint32_t old = atomicAdd(&p.ws.counter[r], 1u);
      last = (old + 1u == need);
    }
    last = __shfl_sync(0xFFFFFFFFu, last, 0);
    if (last) {
      __threadfence();
      if (MODE == MODE_TREE)
        finalize_tree(p, r, s_base[r], len, lane);
      else if (MODE == MODE_CHAIN_GREEDY)
        finalize_chain_greedy<DT>(p, r, s_base[r], len, lane);
      else
        finalize_chain_sample<DT>(p, r, s_base[r], len, lane);
      if (lane == 0) p.ws.counter[r] = 0u;
    }
  }
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
    const Record* recp = reinterpret_cast<const Record*>(p.ws.record) + r;
    const int flag = __ldcg(&recp->flag);
    if (!flag) continue;
    const Record rec = *recp;
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
      double ls = 0.0;
#pragma unroll
      for (int j = 0; j < 64; ++j) ls += (double)resid(vp, vq, j);
      const double ws = warp_sum_d(ls);
      if (lane == 0) __stcg(&p.ws.partial2[(int64_t)r * p.ws.units + u], ws);
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
    // total residual mass; at or below 1e-30 the draw falls back to p
    double Z;
    {
      double ls = 0.0;
      for (int uu = lane; uu < units; uu += 32) ls += __ldcg(&p.ws.partial2[(int64_t)r * p.ws.units + uu]);
      Z = warp_sum_d(ls);
    }
    const bool fallback = !(Z > 1e-30);
    const int pslot = rec.prow;
    auto w_res = [&](int uu) -> double { return __ldcg(&p.ws.partial2[(int64_t)r * p.ws.units + uu]); };
    auto w_p = [&](int uu) -> double {
      const float2 t = __ldcg(&p.ws.partial[(int64_t)pslot * p.ws.units + uu]);
      if (t.x == -INFINITY) return 0.0;
      return (double)(t.y * ex2((t.x - rec.mp) * p.c) * ip);
    };
    Crossing cr;
    double tot;
    if (fallback) {
      tot = find_unit(units, 0.0, lane, w_p).total;
      cr = find_unit(units, (double)rec.u2 * tot, lane, w_p);
    } else {
      tot = Z;
      cr = find_unit(units, (double)rec.u2 * tot, lane, w_res);
    }
    const double t = (double)rec.u2 * tot;
    const int e0 = cr.unit * SPEC_UNIT, n_el = min(SPEC_UNIT, p.vocab - e0);
    float vp[64], vq[64], rr[64];
    load_unit_contig<DT>(prow, e0, n_el, vec, lane, vp);
    load_unit_contig<DT>(qrow, e0, n_el, vec, lane, vq);
#pragma unroll
    for (int j = 0; j < 64; ++j)
      rr[j] = fallback ? (vp[j] == -INFINITY ? 0.0f : ex2(fmaf(vp[j], p.c, -mpc)) * ip) : resid(vp, vq, j);
    float r_at;
    const int pick = find_in_unit(rr, cr.before, t, lane, &r_at);
    if (lane == 0) {
      p.out_tokens[(int64_t)r * (p.L + 1) + rec.pos - 1] = e0 + pick;
      if (p.dbg_resid) p.dbg_resid[r] = (float)((double)r_at / tot);
      Record* wr = reinterpret_cast<Record*>(p.ws.record) + r;
      wr->flag = 0;
      p.ws.counter2[r] = 0u;
    }
  }
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
  const size_t smem = (size_t)(3 * p.batch + 1) * sizeof(int32_t);
  auto k = spec::verify_rows_kernel<DT, MODE>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  static int cached_grid = 0;
  static size_t cached_smem = 0;
  if (cached_grid == 0 || cached_smem != smem) {
    cached_grid = grid_for(k, smem, num_sms);
    cached_smem = smem;
  }
  k<<<cached_grid, SPEC_CTA_THREADS, smem, stream>>>(p);
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
