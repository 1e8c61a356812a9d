// pricing.cuh -- device functions of step 2 (pricing, chain choice, budget
// allocation), shared by the standalone pricing kernel and the fused
// draft-and-price kernel.
//
// Hybrid Spark Algorithm 1 and sec. 4.2-4.5:
//   h_k   Eq. (1), read from a table built once per coefficient set in fp64 and
//         rounded once to fp32 (contiguous in k for one (n, a, m));
//   S^g_k = S^g_{k-1} h_k,  S^d_k = S^d_{k-1} c_k          (fp32, k order)
//   V     = sum_k max(S_k - lambda, 0)                     (Eq. (3), fp32)
//   contains rule / value rule / lossless policies (sec. 4.3, 4.5, App. H)
//   AV allocation: the top-b (request, position) slots by S, ties to the lower
//   request then position; every request keeps a prefix (sec. 2, sec. 4.4).
// Every product and sum is one correctly rounded fp32 operation in a fixed
// order, so the selection is reproducible bit for bit.
#pragma once

#include "common.cuh"

#define SPEC_TAB_N 33  // n in [0, SPEC_MAX_N]

namespace spec {

struct PriceCtx {
  int32_t K, L;
  const float* table;
  int32_t tab_const, n_full, m_cap;
  float lambda;
  int32_t policy, draft_greedy;
  int32_t* chain;
  float* S;
  int32_t* chain_len;
  int32_t* source;
  uint8_t* point_mass;
};

struct SelectCtx {
  int32_t batch, L, budget, mvl;
  const float* S;
  const int32_t* chain_len;
  int32_t* verify_len;
  int32_t* row_off;
};

__device__ __forceinline__ float clamp_conf(float ck, uint32_t& st) {
  if (!(ck >= 0.0f)) {  // negative or NaN
    st |= SPEC_DEV_BAD_VALUE;
    return 0.0f;
  }
  if (ck > 1.0f) {
    st |= SPEC_DEV_BAD_VALUE;
    return 1.0f;
  }
  return ck;
}

// The Eq. (1) table row of features (n, a, m): h_1..h_L contiguous, or null
// when n lies outside the table (h = 0, flagged).
__device__ __forceinline__ const float* table_row(const PriceCtx& cx, int32_t n, int32_t a, int32_t m,
                                                  int32_t gl, uint32_t& st) {
  if (cx.tab_const) return cx.table;
  if (n == cx.n_full) {
    m = m < 0 ? 0 : (m > cx.m_cap ? cx.m_cap : m);
    return cx.table + (int64_t)cx.L * SPEC_TAB_N * 2 + (int64_t)(a * (cx.m_cap + 1) + m) * cx.L;
  }
  if (n >= 0 && n <= SPEC_MAX_N) return cx.table + (int64_t)(n * 2 + a) * cx.L;
  if (gl > 0) st |= SPEC_DEV_BAD_VALUE;
  return nullptr;
}

// Chain choice and survivals of request r by one warp.  Every lane reads the
// request's whole (short) rows -- the same addresses, so one broadcast load per
// element -- and forms the sequential products and sums itself, left to right
// in k, one correctly rounded fp32 operation at a time; lane k then writes
// position k+1.  `gt`/`dt`/`ct` are the n-gram tokens, model tokens and
// confidences (global or shared memory, any lane may read any entry).
__device__ __forceinline__ void price_request_warp(const PriceCtx& cx, int r, int lane, const int32_t* gt,
                                                   int32_t gl, int32_t n, int32_t a, int32_t m,
                                                   const int32_t* dt, const float* ct, int32_t dl,
                                                   uint32_t& st) {
  const int32_t K = cx.K, L = cx.L;
  if (dl < 0 || dl > K) {
    st |= SPEC_DEV_BAD_LENGTH;
    dl = dl < 0 ? 0 : K;
  }
  if (gl < 0 || gl > L) {
    st |= SPEC_DEV_BAD_LENGTH;
    gl = gl < 0 ? 0 : L;
  }
  if (a != 0 && a != 1) {
    st |= SPEC_DEV_BAD_VALUE;
    a = 1;
  }
  const float* hrow = table_row(cx, n, a, m, gl, st);
  float hv[SPEC_MAX_L], cv[SPEC_MAX_L];
  int32_t gv[SPEC_MAX_L], dv[SPEC_MAX_L];
#pragma unroll
  for (int j = 0; j < SPEC_MAX_L; ++j) {
    hv[j] = (j < gl && hrow) ? __ldg(hrow + (cx.tab_const ? 0 : j)) : 0.0f;
    gv[j] = j < gl ? gt[j] : -1;
    dv[j] = j < dl ? dt[j] : -1;
    cv[j] = j < dl ? ct[j] : 0.0f;
  }
  uint32_t st_c = 0;
#pragma unroll
  for (int j = 0; j < SPEC_MAX_L; ++j)
    if (j < dl) cv[j] = clamp_conf(cv[j], st_c);
  if (lane == 0) st |= st_c;
  // survivals and chain values, left to right
  float sg[SPEC_MAX_L], sd[SPEC_MAX_L];
  float run_g = 1.0f, run_d = 1.0f, vg = 0.0f, vd = 0.0f;
  bool d_prefix = dl >= 1 && gl > dl;
#pragma unroll
  for (int j = 0; j < SPEC_MAX_L; ++j) {
    run_g = __fmul_rn(run_g, hv[j]);
    run_d = __fmul_rn(run_d, cv[j]);
    sg[j] = run_g;
    sd[j] = run_d;
    if (j < gl) vg = __fadd_rn(vg, fmaxf(__fsub_rn(run_g, cx.lambda), 0.0f));
    if (j < dl) {
      vd = __fadd_rn(vd, fmaxf(__fsub_rn(run_d, cx.lambda), 0.0f));
      if (gv[j] != dv[j]) d_prefix = false;
    }
  }
  int32_t src = SPEC_SRC_MODEL;
  switch (cx.policy) {
    case SPEC_POLICY_PROPOSED:
      src = d_prefix ? SPEC_SRC_CONTAINS : ((gl > 0 && vg >= vd) ? SPEC_SRC_NGRAM : SPEC_SRC_MODEL);
      break;
    case SPEC_POLICY_NGRAM_FIRST:
      src = gl > 0 ? SPEC_SRC_NGRAM : SPEC_SRC_MODEL;
      break;
    case SPEC_POLICY_EXTENSION:
      src = d_prefix ? SPEC_SRC_EXTENSION : SPEC_SRC_MODEL;
      break;
    case SPEC_POLICY_MODEL_ONLY:
      src = SPEC_SRC_MODEL;
      break;
    default:
      src = SPEC_SRC_NGRAM;
      break;
  }
  const int32_t len = (src == SPEC_SRC_MODEL) ? dl : gl;
  const uint8_t model_pm = cx.draft_greedy ? 1 : 0;
  // lane k emits position k+1 (register arrays are read at constant indices)
  const int k = lane;
  int32_t tok = -1;
  float sv = 0.0f;
  uint8_t pm = 0;
  float prev = 1.0f;
#pragma unroll
  for (int j = 0; j < SPEC_MAX_L; ++j) {
    if (j < len) {
      int32_t tj;
      float sj;
      uint8_t pj;
      if (src == SPEC_SRC_MODEL) {
        tj = dv[j];
        sj = sd[j];
        pj = model_pm;
      } else if (src == SPEC_SRC_NGRAM) {
        tj = gv[j];
        sj = sg[j];
        pj = 1;
      } else {
        // contains rule / extension: the first dl positions take max(S^g, S^d)
        // (contains) or S^d (extension); the tail continues S_j = S_{j-1} h_j
        tj = gv[j];
        if (j < dl) {
          sj = (src == SPEC_SRC_CONTAINS) ? fmaxf(sg[j], sd[j]) : sd[j];
          pj = (src == SPEC_SRC_EXTENSION) ? model_pm : (uint8_t)1;
        } else {
          sj = __fmul_rn(prev, hv[j]);
          pj = 1;
        }
        prev = sj;
      }
      if (j == k) {
        tok = tj;
        sv = sj;
        pm = pj;
      }
    }
  }
  if (k < L) {
    cx.chain[(int64_t)r * L + k] = tok;
    cx.S[(int64_t)r * L + k] = sv;
    cx.point_mass[(int64_t)r * L + k] = pm;
  }
  if (lane == 0) {
    cx.chain_len[r] = len;
    cx.source[r] = src;
  }
}

// ---------------------------------------------------------------------------
// Batch-wide allocation by one CTA (all its threads call this).
// Slot q = r * L + k (request, position order); its key is w = bits(S) + 1 for
// a valid slot (k < min(chain_len, max_verify_len)), 0 otherwise (survivals
// are >= 0, so their bits order like their values, and S <= 1.0f keeps w below
// 2^30).  theta, the budget-th largest survival, is the largest t with
// count(w >= t + 1) >= budget, built two bits per step from the top with one
// barrier per step; slots above theta are taken, then the ties at theta in
// slot order until the budget is spent.
// Shared scratch: select_scratch_ints(batch, L) ints.
__host__ __device__ inline int select_scratch_ints(int batch, int L) { return batch * L + batch + 64; }

static __device__ __forceinline__ int32_t cta_sum(int32_t v, int32_t* red /*[2][32]*/, int& parity) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = __reduce_add_sync(0xFFFFFFFFu, v);
  int32_t* buf = red + 32 * parity;
  if (lane == 0) buf[warp] = v;
  __syncthreads();
  int32_t t = 0;
  const int nw = (blockDim.x + 31) >> 5;
  for (int q = 0; q < nw; ++q) t += buf[q];
  parity ^= 1;  // the next call writes the other buffer: no second barrier
  return t;
}

static __device__ __forceinline__ void select_budget_cta(const SelectCtx& sc, int32_t* scratch) {
  const int B = sc.batch, L = sc.L;
  const int nslots = B * L;
  const int tid = threadIdx.x, nt = blockDim.x;
  uint32_t* s_key = reinterpret_cast<uint32_t*>(scratch);  // [nslots]
  int32_t* s_ell = scratch + nslots;                        // [B]
  int32_t* red = s_ell + B;                                 // [64]
  int parity = 0;
  // keys: batches of 8 slots per thread, every load issued before any is used
  int32_t my_valid = 0;
  for (int q0 = 0; q0 < nslots; q0 += 8 * nt) {
    float sv[8];
    int32_t len[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int q = q0 + tid + i * nt;
      sv[i] = q < nslots ? __ldcg(sc.S + q) : 0.0f;
      len[i] = q < nslots ? __ldcg(sc.chain_len + q / L) : 0;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int q = q0 + tid + i * nt;
      if (q < nslots) {
        const int k = q - (q / L) * L;
        const bool valid = k < len[i] && k < sc.mvl;
        s_key[q] = valid ? __float_as_uint(sv[i]) + 1u : 0u;
        my_valid += valid;
      }
    }
  }
  for (int r = tid; r < B; r += nt) s_ell[r] = 0;
  const int32_t n_valid = cta_sum(my_valid, red, parity);  // (its barrier orders the stores above)
  const int32_t budget = sc.budget;
  if (budget >= n_valid || budget == 0) {
    for (int r = tid; r < B; r += nt) {
      const int32_t len = __ldcg(sc.chain_len + r);
      s_ell[r] = budget > 0 ? (len < sc.mvl ? len : sc.mvl) : 0;
    }
  } else {
    uint32_t t = 0u;  // bits of theta, two at a time from bit 29
    for (int shift = 28; shift >= 0; shift -= 2) {
      const uint32_t c1 = (t | (1u << shift)) + 1u, c2 = (t | (2u << shift)) + 1u, c3 = (t | (3u << shift)) + 1u;
      int32_t n1 = 0, n2 = 0, n3 = 0;
      for (int q = tid; q < nslots; q += nt) {
        const uint32_t w = s_key[q];
        n1 += w >= c1;
        n2 += w >= c2;
        n3 += w >= c3;
      }
      n1 = __reduce_add_sync(0xFFFFFFFFu, n1);
      n2 = __reduce_add_sync(0xFFFFFFFFu, n2);
      n3 = __reduce_add_sync(0xFFFFFFFFu, n3);
      int32_t* buf = red + 32 * parity;
      const int lane = tid & 31, warp = tid >> 5;
      if (lane == 0) {
        buf[warp] = n1;
        buf[warp + 8] = n2;
        buf[warp + 16] = n3;
      }
      __syncthreads();
      int32_t m1 = 0, m2 = 0, m3 = 0;
      for (int q = 0; q < (nt >> 5); ++q) {
        m1 += buf[q];
        m2 += buf[q + 8];
        m3 += buf[q + 16];
      }
      parity ^= 1;
      const uint32_t j = m3 >= budget ? 3u : (m2 >= budget ? 2u : (m1 >= budget ? 1u : 0u));
      t |= j << shift;
    }
    const uint32_t key_eq = t + 1u;
    int32_t above = 0;
    for (int q = tid; q < nslots; q += nt) above += s_key[q] > key_eq;
    const int32_t need = budget - cta_sum(above, red, parity);  // ties at theta to take
    // ties in slot order: contiguous slot ranges per thread, one block scan
    const int per = (nslots + nt - 1) / nt;
    const int q_lo = tid * per, q_hi = min(nslots, q_lo + per);
    int32_t eq = 0;
    for (int q = q_lo; q < q_hi; ++q) eq += s_key[q] == key_eq;
    const int lane = tid & 31, warp = tid >> 5;
    int32_t incl = eq;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += v;
    }
    int32_t* buf = red + 32 * parity;
    if (lane == 31) buf[warp] = incl;
    __syncthreads();
    int32_t rank = incl - eq;
    for (int q = 0; q < warp; ++q) rank += buf[q];
    int cur_r = -1, cur_n = 0;
    for (int q = q_lo; q < q_hi; ++q) {
      const uint32_t w = s_key[q];
      const bool sel = w > key_eq || (w == key_eq && rank++ < need);
      if (sel) {
        const int r = q / L;
        if (r != cur_r) {
          if (cur_n) atomicAdd(&s_ell[cur_r], cur_n);
          cur_r = r;
          cur_n = 0;
        }
        ++cur_n;
      }
    }
    if (cur_n) atomicAdd(&s_ell[cur_r], cur_n);
    parity ^= 1;
  }
  __syncthreads();
  // row offsets: contiguous request ranges per thread, one block scan
  const int rp = (B + nt - 1) / nt;
  const int r_lo = tid * rp, r_hi = min(B, r_lo + rp);
  int32_t mine = 0;
  for (int r = r_lo; r < r_hi; ++r) mine += s_ell[r] + 1;
  const int lane = tid & 31, warp = tid >> 5;
  int32_t incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += v;
  }
  int32_t* buf = red + 32 * parity;
  if (lane == 31) buf[warp] = incl;
  __syncthreads();
  int32_t off = incl - mine, total = 0;
  for (int q = 0; q < (nt >> 5); ++q) {
    if (q < warp) off += buf[q];
    total += buf[q];
  }
  for (int r = r_lo; r < r_hi; ++r) {
    sc.verify_len[r] = s_ell[r];
    sc.row_off[r] = off;
    off += s_ell[r] + 1;
  }
  if (tid == 0) sc.row_off[B] = total;
}

}  // namespace spec
