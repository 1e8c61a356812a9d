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
#define SPEC_TAB_SMEM_MAX (48 * 1024)  // the largest Eq. (1) table fused pricing stages in shared memory

namespace spec {

struct PriceCtx {
  int32_t K, L;
  const float* table;
  int32_t tab_const, n_full, m_cap;
  float lambda;
  int32_t policy, draft_greedy, mvl;
  int32_t* chain;
  float* S;
  int32_t* chain_len;
  int32_t* source;
  uint8_t* point_mass;
  uint32_t* keys;  // [batch x L] allocation keys (workspace)
};

struct SelectCtx {
  int32_t batch, L, budget;
  const uint32_t* keys;
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
__device__ __forceinline__ const float* table_row(const PriceCtx& cx, const float* table, int32_t n, int32_t a,
                                                  int32_t m, int32_t gl, uint32_t& st) {
  if (cx.tab_const) return table;
  if (n == cx.n_full) {
    m = m < 0 ? 0 : (m > cx.m_cap ? cx.m_cap : m);
    return table + (int64_t)cx.L * SPEC_TAB_N * 2 + (int64_t)(a * (cx.m_cap + 1) + m) * cx.L;
  }
  if (n >= 0 && n <= SPEC_MAX_N) return table + (int64_t)(n * 2 + a) * cx.L;
  if (gl > 0) st |= SPEC_DEV_BAD_VALUE;
  return nullptr;
}

// One request's short rows, staged in shared memory by the warp that prices it.
struct PriceStage {
  float h[32];    // h_1..h_gl (filled by price_request_warp)
  int32_t g[32];  // n-gram chain
  int32_t d[32];  // model drafter's chain
  float c[32];    // model drafter's confidences (clamped in place)
};

// Chain choice, survivals and allocation keys of request r by one warp (all 32
// lanes call it).  On entry ps.g[0, min(gl, L)), ps.d[0, K) and ps.c[0, K) hold
// the request's n-gram tokens, model tokens and raw confidences, written by
// this warp before a __syncwarp.  Lane j stages h_{j+1}; then every lane runs
// the same left-to-right recurrence over the staged rows, one correctly
// rounded fp32 operation at a time, and keeps the values of position j+1,
// which it writes.  The loops are unrolled by four, so that the staged values
// of four positions are loaded together ahead of the dependent products: this
// code runs once per request, and its latency is on the critical path of the
// round.
// stab: a copy of the Eq. (1) table in this CTA's shared memory, or null to
// read the table in global memory.
__device__ __forceinline__ int32_t price_request_warp(const PriceCtx& cx, int r, int lane, PriceStage& ps,
                                                   int32_t gl, int32_t n, int32_t a, int32_t m, int32_t dl,
                                                   uint32_t& st, const float* stab) {
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
  const float* hrow = table_row(cx, stab ? stab : cx.table, n, a, m, gl, st);
  if (lane < gl) {
    const float* hp = hrow + (cx.tab_const ? 0 : lane);
    ps.h[lane] = hrow ? (stab ? *hp : __ldg(hp)) : 0.0f;
  }
  if (lane < dl) ps.c[lane] = clamp_conf(ps.c[lane], st);
  __syncwarp();
  // S^g_k, S^d_k and the chain values, k = 1, 2, ... in order
  float run_g = 1.0f, run_d = 1.0f, vg = 0.0f, vd = 0.0f, my_g = 0.0f, my_d = 0.0f;
  bool d_prefix = dl >= 1 && gl > dl;  // d is a proper prefix of g (contains rule)
  const int32_t jn = gl > dl ? gl : dl;
#pragma unroll 4
  for (int j = 0; j < jn; ++j) {
    if (j < gl) {
      run_g = __fmul_rn(run_g, ps.h[j]);
      vg = __fadd_rn(vg, fmaxf(__fsub_rn(run_g, cx.lambda), 0.0f));
      if (j == lane) my_g = run_g;
    }
    if (j < dl) {
      run_d = __fmul_rn(run_d, ps.c[j]);
      vd = __fadd_rn(vd, fmaxf(__fsub_rn(run_d, cx.lambda), 0.0f));
      if (j == lane) my_d = run_d;
      d_prefix = d_prefix && ps.g[j] == ps.d[j];
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
  int32_t tok = -1;
  float sv = 0.0f;
  uint8_t pm = 0;
  if (src == SPEC_SRC_MODEL) {
    if (lane < dl) {
      tok = ps.d[lane];
      sv = my_d;
      pm = model_pm;
    }
  } else if (src == SPEC_SRC_NGRAM) {
    if (lane < gl) {
      tok = ps.g[lane];
      sv = my_g;
      pm = 1;
    }
  } else {
    // contains rule / extension: the first dl positions take max(S^g, S^d)
    // (contains) or S^d (extension); the tail continues S_j = S_{j-1} h_j
    const bool contains = (src == SPEC_SRC_CONTAINS);
    if (lane < gl) tok = ps.g[lane];
    if (lane < dl) {
      sv = contains ? fmaxf(my_g, my_d) : my_d;
      pm = contains ? (uint8_t)1 : model_pm;
    }
    float prev = __shfl_sync(0xFFFFFFFFu, sv, dl - 1);  // dl >= 1 on this branch
#pragma unroll 4
    for (int j = dl; j < gl; ++j) {
      prev = __fmul_rn(prev, ps.h[j]);
      if (j == lane) {
        sv = prev;
        pm = 1;
      }
    }
  }
  if (lane < L) {
    const int64_t q = (int64_t)r * L + lane;
    cx.chain[q] = tok;
    cx.S[q] = sv;
    cx.point_mass[q] = pm;
    // allocation key: survival bits + 1 for a slot that may be verified, 0
    // otherwise (S >= 0, so the bits order like the values; S <= 1 keeps the
    // key below 2^30)
    cx.keys[q] = (lane < len && lane < cx.mvl) ? __float_as_uint(sv) + 1u : 0u;
  }
  if (lane == 0) {
    cx.chain_len[r] = len;
    cx.source[r] = src;
  }
  return len;
}

// ---------------------------------------------------------------------------
// Batch-wide allocation by one CTA of exactly 256 threads (all call this).
// Slot q = r * L + k is taken when its key exceeds theta, or equals theta and
// lies among the first `need` such slots in slot order; theta and need follow
// from the budget: none (theta = ~0), every valid slot (budget >= number of
// valid slots: theta = 0), else theta = the key of the budget-th slot in the
// order (key desc, slot asc).  A 1024-bin shared-memory histogram of the
// survival value (linear bins) locates it (then of key bits 29..20, 19..10,
// 9..0 among that bin's keys while the chosen bin still holds more than 256
// keys), and the keys of the chosen bin are then ranked against each other
// directly.  Survivals fall
// along a chain (products of factors in [0, 1]) and ties go to the lower
// position, so every request takes a prefix:
// ell_r = above_r + min(eq_r, max(0, need - E_r)) with E_r the ties of the
// requests before r, and row_off[r] = r + sum_{r' < r} above_r' + min(need, E_r),
// one block scan of the pair (above, eq).
// The histogram and candidate passes over the keys are rolled loops: one CTA
// runs this once per launch, on an SM whose instruction cache holds other
// code by then (in a decode step the verification kernel runs between two
// launches), so fewer instruction lines count for more there than iterations
// in flight.  The ranking and the per-request counts keep four iterations in
// flight: rolled, their dependent shared-memory reads add up.
// Shared scratch: select_scratch_ints(batch, L) ints.
__host__ __device__ inline int select_scratch_ints(int batch, int L) {
  return ((batch * L + 3) & ~3) + 2 * 1024 + 256 + 96;
}

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

// inclusive prefix sum over the CTA in thread order; *total gets the sum
static __device__ __forceinline__ int32_t cta_incl_scan(int32_t v, int32_t* red, int& parity, int32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int32_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += t;
  }
  int32_t* buf = red + 32 * parity;
  if (lane == 31) buf[warp] = incl;
  __syncthreads();
  int32_t before = 0, all = 0;
  const int nw = (blockDim.x + 31) >> 5;
  for (int q = 0; q < nw; ++q) {
    const int32_t b = buf[q];
    before += q < warp ? b : 0;
    all += b;
  }
  parity ^= 1;
  *total = all;
  return incl + before;
}

static __device__ __forceinline__ void select_budget_cta(const SelectCtx& sc, int32_t* scratch,
                                                         const int32_t* counts = nullptr) {
  constexpr int NB = 1024;   // histogram bins (10 key bits per level)
  constexpr int NCAND = 256; // keys ranked directly
  const int B = sc.batch, L = sc.L;
  const int nslots = B * L;
  const int tid = threadIdx.x, nt = blockDim.x;
  // At most 32 requests: warp 0 counts each request's valid slots (lane r,
  // request r; from `counts` when the caller has them, else from the keys).  A budget of zero or one that covers every valid slot decides
  // every length at once (all valid slots, or none), and the warp writes the
  // lengths and offsets itself; the block-wide selection runs otherwise.
  if (B <= 32) {
    __shared__ int32_t s_done;
    if (tid < 32) {
      int32_t cnt = 0;
      if (tid < B) {
        if (counts) {
          cnt = counts[tid];
        } else {
#pragma unroll 4
          for (int k = 0; k < L; ++k) cnt += __ldcg(sc.keys + tid * L + k) != 0u;
        }
      }
      const int32_t n_valid = __reduce_add_sync(0xFFFFFFFFu, cnt);
      const bool done = sc.budget == 0 || sc.budget >= n_valid;
      if (done) {
        const int32_t len = sc.budget == 0 ? 0 : cnt;  // lanes past B hold 0
        int32_t incl = len;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int32_t t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
          if (tid >= o) incl += t;
        }
        if (tid < B) {
          sc.verify_len[tid] = len;
          sc.row_off[tid] = tid + incl - len;
        }
        if (tid == 31) sc.row_off[B] = B + incl;
      }
      if (tid == 0) s_done = done ? 1 : 0;
    }
    __syncthreads();
    if (s_done) return;
  }
  uint32_t* s_key = reinterpret_cast<uint32_t*>(scratch);          // [nslots]
  int32_t* s_hist = scratch + ((nslots + 3) & ~3);                  // [2][NB], 16-byte aligned
  uint32_t* s_cand = reinterpret_cast<uint32_t*>(s_hist + 2 * NB);  // [NCAND]
  int32_t* red = reinterpret_cast<int32_t*>(s_cand + NCAND);        // [2][32]
  int32_t* bc = red + 64;                                           // [2][4] + candidate count
  int parity = 0;
  for (int i = tid; i < 2 * NB; i += nt) s_hist[i] = 0;
  for (int i = tid; i < NCAND; i += nt) s_cand[i] = 0u;  // the ranking reads whole groups of four
  if (tid == 0) bc[8] = 0;
  // Level 0 of the selection bins the survival value linearly (a valid key is
  // the value's bits + 1, and value x 1024 is exact, so the bins keep the keys'
  // order): keys close in value spread over many bins, and few share the
  // chosen one.
  auto vbin = [](uint32_t w) -> int { return min(NB - 1, (int)(__uint_as_float(w - 1u) * (float)NB)); };
  // keys: batches of 8 slots per thread, every load issued before any is used;
  // with at most 8 per thread they stay in registers (wk) for the candidates
  const bool regs = nslots <= 8 * nt;
  uint32_t wk[8];
  int32_t my_valid = 0;
  for (int q0 = 0; q0 < nslots; q0 += 8 * nt) {
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int q = q0 + tid + i * nt;
      w[i] = q < nslots ? __ldcg(sc.keys + q) : 0u;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int q = q0 + tid + i * nt;
      if (q < nslots) s_key[q] = w[i];
      my_valid += w[i] != 0u;
      wk[i] = w[i];
    }
  }
  const int32_t n_valid = cta_sum(my_valid, red, parity);  // (its barrier orders the stores above)
  const int32_t budget = sc.budget;
  uint32_t theta;
  int32_t need;
  if (budget == 0) {
    theta = 0xFFFFFFFFu;
    need = 0;
  } else if (budget >= n_valid) {
    theta = 0u;
    need = 0;
  } else {
    // Level 0: the value bins.  Only when the chosen bin still holds more than
    // NCAND keys do the next levels fix the key's bits ten at a time among the
    // bin's keys.
    int vb = -1;           // the chosen value bin
    uint32_t prefix = 0u;  // key bits at and above `hi` fixed so far (levels 1..3)
    int hi = 30;           // keys are below 2^30
    int32_t rem = budget;  // slots still to take among the keys of the bin and prefix
    int32_t cnt = nslots;
    auto member = [&](uint32_t w) -> bool { return w != 0u && vbin(w) == vb && (w >> hi) == (prefix >> hi); };
#pragma unroll 1
    for (int level = 0; level < 4; ++level) {
      const int shift = hi - 10;
      int32_t* hist = s_hist + (level & 1) * NB;
#pragma unroll 1
      for (int q = tid; q < nslots; q += nt) {
        const uint32_t w = s_key[q];
        if (level == 0) {
          if (w != 0u) atomicAdd(&hist[vbin(w)], 1);
        } else if (member(w)) {
          atomicAdd(&hist[(w >> shift) & (NB - 1)], 1);
        }
      }
      __syncthreads();
      // thread t owns bins 1023 - 4t .. 1020 - 4t (descending) and zeroes them
      // for the level after next
      const int base = NB - 4 - 4 * tid;
      const int4 h4 = *reinterpret_cast<const int4*>(hist + base);
      *reinterpret_cast<int4*>(hist + base) = make_int4(0, 0, 0, 0);
      const int32_t c4 = h4.x + h4.y + h4.z + h4.w;
      int32_t tot;
      const int32_t incl = cta_incl_scan(c4, red, parity, &tot);
      int32_t e = incl - c4;
      int32_t* b = bc + 4 * (level & 1);
      if (e < rem && incl >= rem) {
        int dg = base + 3;
        int32_t c = h4.w;
        if (e + c < rem) {
          e += c;
          dg = base + 2;
          c = h4.z;
          if (e + c < rem) {
            e += c;
            dg = base + 1;
            c = h4.y;
            if (e + c < rem) {
              e += c;
              dg = base;
              c = h4.x;
            }
          }
        }
        b[0] = dg;
        b[1] = rem - e;
        b[2] = c;
      }
      __syncthreads();
      if (level == 0) {
        vb = b[0];
      } else {
        prefix |= (uint32_t)b[0] << shift;
        hi = shift;
      }
      rem = b[1];
      cnt = b[2];
      if (cnt <= NCAND || hi == 0) break;
    }
    if (hi == 0) {
      // every key bit fixed: the bin holds copies of one key
      theta = prefix;
      need = rem;
    } else {
      // the chosen bin's keys, ranked directly: theta is the value v with
      // #(keys > v) < rem <= #(keys >= v)
      if (regs) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (tid + i * nt < nslots && member(wk[i])) s_cand[atomicAdd(&bc[8], 1)] = wk[i];
      } else {
#pragma unroll 1
        for (int q = tid; q < nslots; q += nt) {
          const uint32_t w = s_key[q];
          if (member(w)) s_cand[atomicAdd(&bc[8], 1)] = w;
        }
      }
      __syncthreads();
      int32_t* b = bc + 4 * 2;  // words 8..11: [8] count (done), [9] theta, [10] need
      if (tid < cnt) {
        // the candidates four at a time (the zeroes past cnt count in neither
        // sum: the key sought is at least 1)
        const uint32_t v = s_cand[tid];
        const uint4* c4 = reinterpret_cast<const uint4*>(s_cand);
        int32_t gt = 0, ge = 0;
#pragma unroll 4
        for (int i = 0; i < ((cnt + 3) >> 2); ++i) {
          const uint4 u = c4[i];
          gt += (int32_t)(u.x > v) + (int32_t)(u.y > v) + (int32_t)(u.z > v) + (int32_t)(u.w > v);
          ge += (int32_t)(u.x >= v) + (int32_t)(u.y >= v) + (int32_t)(u.z >= v) + (int32_t)(u.w >= v);
        }
        if (gt < rem && rem <= ge) {  // every copy of v writes the same values
          b[1] = (int32_t)v;
          b[2] = rem - gt;
        }
      }
      __syncthreads();
      theta = (uint32_t)b[1];
      need = b[2];
    }
  }
  // per request: slots above theta and ties at theta; contiguous request
  // ranges per thread, packed (above << 16 | eq): each is at most
  // 1024 x 31 slots, so neither field overflows
  const int rp = (B + nt - 1) / nt;
  const int r_lo = min(B, tid * rp), r_hi = min(B, r_lo + rp);
  int32_t mine = 0, above0 = 0, eq0 = 0;  // (above, eq) of request r_lo, kept for the second pass
  for (int r = r_lo; r < r_hi; ++r) {
    int32_t above = 0, eq = 0;
#pragma unroll 4
    for (int k = 0; k < L; ++k) {
      const uint32_t w = s_key[r * L + k];
      above += w > theta;
      eq += w == theta;
    }
    if (r == r_lo) {
      above0 = above;
      eq0 = eq;
    }
    mine += (above << 16) | eq;
  }
  int32_t tot;
  const int32_t incl = cta_incl_scan(mine, red, parity, &tot);
  int32_t A = (incl - mine) >> 16, E = (incl - mine) & 0xFFFF;
  for (int r = r_lo; r < r_hi; ++r) {
    int32_t above = above0, eq = eq0;
    if (r != r_lo) {
      above = 0;
      eq = 0;
#pragma unroll 4
      for (int k = 0; k < L; ++k) {
        const uint32_t w = s_key[r * L + k];
        above += w > theta;
        eq += w == theta;
      }
    }
    const int32_t take = min(eq, max(0, need - E));
    sc.verify_len[r] = above + take;
    sc.row_off[r] = r + A + min(need, E);
    A += above;
    E += eq;
  }
  if (tid == 0) sc.row_off[B] = B + (tot >> 16) + min(need, tot & 0xFFFF);
}

}  // namespace spec
