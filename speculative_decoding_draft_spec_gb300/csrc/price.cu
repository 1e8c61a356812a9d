// price.cu -- step 2 of the round: pricing, chain choice, budget allocation.
//
// Hybrid Spark Algorithm 1 and sec. 4.2-4.5:
//   h_k   Eq. (1), read from a table built once per coefficient set in fp64
//         (estimator_table_kernel) and rounded once to fp32;
//   S^g_k = S^g_{k-1} h_k,  S^d_k = S^d_{k-1} c_k          (fp32, k order)
//   V     = sum_k max(S_k - lambda, 0)                     (Eq. (3), fp32)
//   contains rule / value rule / lossless policies (sec. 4.3, 4.5, App. H)
//   AV allocation: the top-b (request, position) slots by S, ties to the lower
//   request then position; every request keeps a prefix (sec. 2, sec. 4.4).
// All products and sums use explicit round-to-nearest intrinsics in a fixed
// order so that the selection is reproducible bit for bit.
//
// GB300 layout: one CTA of up to 1024 threads, one thread per request for the
// per-request arithmetic; survivals staged in shared memory ([L][batch], so
// consecutive threads touch consecutive banks); the b-th largest survival is
// found by a 4-pass 8-bit radix select over the fp32 bit patterns (survivals
// are non-negative, so their bits order like their values) with shared-memory
// histograms; ties at the threshold are resolved in (request, position) order
// by a block-wide exclusive scan; a second scan builds the row offsets.
#include "common.cuh"

namespace spec {

// ------------------------------------------------------------------ Eq. (1)
struct EstimatorDev {
  double beta[32];
  double w_first, w_rest, delta, ell_first, ell_rest, kappa_first, kappa_rest;
  int32_t n_ref, n_full, m_cap, m_ref, use_constant_h;
  double constant_h;
};

#define SPEC_TAB_N 33  // n in [0, SPEC_MAX_N]

__host__ __device__ inline int64_t table_entries(int32_t L, int32_t m_cap, int32_t constant) {
  return constant ? 1 : (int64_t)L * SPEC_TAB_N * 2 + (int64_t)L * 2 * (m_cap + 1);
}

__global__ void estimator_table_kernel(EstimatorDev e, int32_t L, float* table) {
  const int64_t partA = (int64_t)L * SPEC_TAB_N * 2;
  const int64_t total = table_entries(L, e.m_cap, e.use_constant_h);
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    if (e.use_constant_h) {
      table[idx] = __double2float_rn(e.constant_h);
      continue;
    }
    int32_t k, n, a, m;
    bool full;
    if (idx < partA) {
      k = (int32_t)(idx / (SPEC_TAB_N * 2)) + 1;
      n = (int32_t)((idx / 2) % SPEC_TAB_N);
      a = (int32_t)(idx % 2);
      m = n;
      full = false;
    } else {
      const int64_t j = idx - partA;
      const int64_t per_k = 2 * (int64_t)(e.m_cap + 1);
      k = (int32_t)(j / per_k) + 1;
      a = (int32_t)((j / (e.m_cap + 1)) % 2);
      m = (int32_t)(j % (e.m_cap + 1));
      n = e.n_full;
      full = true;
    }
    const bool first = (k == 1);
    double z = e.beta[k - 1];
    z = __dadd_rn(z, __dmul_rn(first ? e.w_first : e.w_rest, (double)(n - e.n_ref)));
    z = __dadd_rn(z, __dmul_rn(e.delta, (double)a));
    if (full) {
      const int32_t mm = m < e.m_cap ? m : e.m_cap;
      double bonus = first ? e.ell_first : e.ell_rest;
      bonus = __dadd_rn(bonus, __dmul_rn(first ? e.kappa_first : e.kappa_rest,
                                         log(__ddiv_rn((double)mm, (double)e.m_ref))));
      z = __dadd_rn(z, bonus);
    }
    const double h = __ddiv_rn(1.0, __dadd_rn(1.0, exp(-z)));
    table[idx] = __double2float_rn(h);
  }
}

// ------------------------------------------------------------------ pricing
struct PriceParams {
  int32_t batch, K, L;
  const int32_t* d;
  const float* c;
  const int32_t* d_len;
  const int32_t* g;
  const int32_t* g_len;
  const int32_t* match_n;
  const int32_t* agree;
  const int32_t* copy_len;
  const float* table;
  int32_t tab_const, n_full, m_cap;
  float lambda;
  int32_t budget, mvl, policy, draft_greedy;
  int32_t* chain;
  float* S;
  int32_t* chain_len;
  int32_t* source;
  int32_t* verify_len;
  int32_t* row_off;
  uint8_t* point_mass;
  uint32_t* status;
};

struct Feat {
  int32_t n, a, m;
  bool tab_ok;
};

__device__ __forceinline__ float lookup_h(const PriceParams& p, const Feat& f, int32_t k /*0-based*/) {
  if (p.tab_const) return __ldg(p.table);
  if (!f.tab_ok) return 0.0f;
  if (f.n == p.n_full) {
    const int64_t off = (int64_t)p.L * SPEC_TAB_N * 2 +
                        ((int64_t)(k * 2 + f.a) * (p.m_cap + 1)) + f.m;
    return __ldg(p.table + off);
  }
  return __ldg(p.table + ((int64_t)k * SPEC_TAB_N + f.n) * 2 + f.a);
}

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

// block-wide exclusive scan of one int per thread (blockDim.x <= 1024)
__device__ int32_t block_excl_scan(int32_t v, int32_t* sh_warp, int32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t t = __shfl_up_sync(0xFFFFFFFFu, x, o);
    if (lane >= o) x += t;
  }
  if (lane == 31) sh_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    const int nw = (blockDim.x + 31) >> 5;
    int32_t y = lane < nw ? sh_warp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t t = __shfl_up_sync(0xFFFFFFFFu, y, o);
      if (lane >= o) y += t;
    }
    if (lane < nw) sh_warp[lane] = y;  // inclusive warp totals
    if (lane == 31) *total = y;
  }
  __syncthreads();
  const int32_t before = warp > 0 ? sh_warp[warp - 1] : 0;
  const int32_t out = before + x - v;
  __syncthreads();
  return out;
}

__global__ void __launch_bounds__(1024) price_kernel(PriceParams p) {
  extern __shared__ __align__(16) float s_S[];  // [L][batch]
  __shared__ int32_t sh_warp[32];
  __shared__ int32_t sh_total;
  __shared__ uint32_t hist[256];
  __shared__ uint32_t sh_prefix, sh_need;

  const int r = threadIdx.x;
  const bool active = r < p.batch;
  uint32_t st = 0;
  int32_t lim = 0;

  if (active) {
    const int32_t K = p.K, L = p.L;
    int32_t dl = p.d_len[r], gl = p.g_len[r];
    if (dl < 0 || dl > K) {
      st |= SPEC_DEV_BAD_LENGTH;
      dl = dl < 0 ? 0 : K;
    }
    if (gl < 0 || gl > L) {
      st |= SPEC_DEV_BAD_LENGTH;
      gl = gl < 0 ? 0 : L;
    }
    Feat f;
    f.n = p.match_n[r];
    f.a = p.agree[r];
    f.m = p.copy_len[r];
    f.tab_ok = true;
    if (f.a != 0 && f.a != 1) {
      st |= SPEC_DEV_BAD_VALUE;
      f.a = 1;
    }
    if (gl > 0 && !p.tab_const) {
      if (f.n == p.n_full) {
        f.m = f.m < 0 ? 0 : (f.m > p.m_cap ? p.m_cap : f.m);
      } else if (f.n < 0 || f.n > SPEC_MAX_N) {
        st |= SPEC_DEV_BAD_VALUE;
        f.tab_ok = false;
      }
    }
    const int32_t* dr = p.d + (int64_t)r * K;
    const int32_t* gr = p.g + (int64_t)r * L;
    const float* cr = p.c + (int64_t)r * K;

    // pass 1: chain values and the contains test
    bool d_prefix = (dl >= 1 && gl > dl);
    float run = 1.0f, vg = 0.0f;
    for (int32_t k = 0; k < gl; ++k) {
      run = __fmul_rn(run, lookup_h(p, f, k));
      const float t = __fsub_rn(run, p.lambda);
      if (t > 0.0f) vg = __fadd_rn(vg, t);
      if (k < dl && gr[k] != dr[k]) d_prefix = false;
    }
    run = 1.0f;
    float vd = 0.0f;
    for (int32_t k = 0; k < dl; ++k) {
      run = __fmul_rn(run, clamp_conf(cr[k], st));
      const float t = __fsub_rn(run, p.lambda);
      if (t > 0.0f) vd = __fadd_rn(vd, t);
    }
    int32_t src = SPEC_SRC_MODEL;
    switch (p.policy) {
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
    // pass 2: the chosen chain, its survivals and point-mass flags
    const int32_t len = (src == SPEC_SRC_MODEL) ? dl : gl;
    float sg = 1.0f, sd = 1.0f, prev = 1.0f;
    const uint8_t model_pm = p.draft_greedy ? 1 : 0;
    for (int32_t k = 0; k < L; ++k) {
      int32_t tok = -1;
      float s = 0.0f;
      uint8_t pm = 0;
      if (k < len) {
        const bool has_g = k < gl, has_d = k < dl;
        const float hk = has_g ? lookup_h(p, f, k) : 0.0f;
        if (has_g) sg = __fmul_rn(sg, hk);
        if (has_d) sd = __fmul_rn(sd, clamp_conf(cr[k], st));
        if (src == SPEC_SRC_MODEL) {
          tok = dr[k];
          s = sd;
          pm = model_pm;
        } else if (src == SPEC_SRC_NGRAM) {
          tok = gr[k];
          s = sg;
          pm = 1;
        } else if (src == SPEC_SRC_CONTAINS) {
          tok = gr[k];
          s = has_d ? fmaxf(sg, sd) : __fmul_rn(prev, hk);
          pm = 1;
        } else {  // extension
          tok = gr[k];
          s = has_d ? sd : __fmul_rn(prev, hk);
          pm = has_d ? model_pm : (uint8_t)1;
        }
        prev = s;
      }
      p.chain[(int64_t)r * L + k] = tok;
      p.S[(int64_t)r * L + k] = s;
      p.point_mass[(int64_t)r * L + k] = pm;
      s_S[k * p.batch + r] = s;
    }
    p.chain_len[r] = len;
    p.source[r] = src;
    lim = len < p.mvl ? len : p.mvl;
  }
  if (st) set_status(p.status, st);
  __syncthreads();

  // ---- top-b threshold: the budget-th largest survival (with multiplicity)
  const int32_t n_valid_excl = block_excl_scan(lim, sh_warp, &sh_total);
  (void)n_valid_excl;
  const int32_t n_valid = sh_total;
  int32_t ell = 0;
  if (p.budget >= n_valid) {
    ell = lim;
  } else if (p.budget > 0) {
    if (threadIdx.x == 0) {
      sh_prefix = 0u;
      sh_need = (uint32_t)p.budget;
    }
    uint32_t mask = 0u;
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0u;
      __syncthreads();
      const uint32_t prefix = sh_prefix;
      if (active)
        for (int32_t k = 0; k < lim; ++k) {
          const uint32_t v = __float_as_uint(s_S[k * p.batch + r]);
          if ((v & mask) == prefix) atomicAdd(&hist[(v >> shift) & 255u], 1u);
        }
      __syncthreads();
      if (threadIdx.x < 32) {
        // lane l owns digits 255-8l .. 248-8l (descending), so lane order is digit order
        const int lane = threadIdx.x;
        uint32_t cnt[8], sum = 0;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          cnt[q] = hist[255 - 8 * lane - q];
          sum += cnt[q];
        }
        uint32_t incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
          if (lane >= o) incl += t;
        }
        const uint32_t need = sh_need;
        const uint32_t excl = incl - sum;
        const bool mine = excl < need && need <= incl;
        if (mine) {
          uint32_t acc = excl;
          for (int q = 0; q < 8; ++q) {
            if (acc + cnt[q] >= need) {
              sh_prefix = prefix | ((uint32_t)(255 - 8 * lane - q) << shift);
              sh_need = need - acc;
              break;
            }
            acc += cnt[q];
          }
        }
      }
      mask |= 255u << shift;
      __syncthreads();
    }
    const uint32_t theta = sh_prefix;
    const int32_t need = (int32_t)sh_need;  // slots equal to theta still to take
    int32_t gt = 0, eq = 0;
    if (active)
      for (int32_t k = 0; k < lim; ++k) {
        const uint32_t v = __float_as_uint(s_S[k * p.batch + r]);
        gt += v > theta;
        eq += v == theta;
      }
    const int32_t eq_before = block_excl_scan(eq, sh_warp, &sh_total);
    int32_t take = need - eq_before;
    take = take < 0 ? 0 : (take > eq ? eq : take);
    ell = gt + take;
  }
  if (active) p.verify_len[r] = ell;
  const int32_t off = block_excl_scan(active ? ell + 1 : 0, sh_warp, &sh_total);
  if (active) p.row_off[r] = off;
  if (threadIdx.x == 0) p.row_off[p.batch] = sh_total;
}

}  // namespace spec

// ---------------------------------------------------------------------------
// host launchers (called from api.cu)
// ---------------------------------------------------------------------------
extern "C" size_t spec_estimator_entries(const spec_estimator* e, int32_t L) {
  return (size_t)spec::table_entries(L, e->m_cap, e->use_constant_h);
}

extern "C" cudaError_t spec_launch_estimator_table(const spec_estimator* e, int32_t L, float* table,
                                                   cudaStream_t stream) {
  spec::EstimatorDev d;
  for (int i = 0; i < 32; ++i) d.beta[i] = e->beta[i];
  d.w_first = e->w_first;
  d.w_rest = e->w_rest;
  d.delta = e->delta;
  d.ell_first = e->ell_first;
  d.ell_rest = e->ell_rest;
  d.kappa_first = e->kappa_first;
  d.kappa_rest = e->kappa_rest;
  d.n_ref = e->n_ref;
  d.n_full = e->n_full;
  d.m_cap = e->m_cap;
  d.m_ref = e->m_ref;
  d.use_constant_h = e->use_constant_h;
  d.constant_h = e->constant_h;
  const int64_t n = spec::table_entries(L, e->m_cap, e->use_constant_h);
  const int threads = 256;
  const int blocks = (int)((n + threads - 1) / threads);
  spec::estimator_table_kernel<<<blocks, threads, 0, stream>>>(d, L, table);
  return cudaGetLastError();
}

extern "C" cudaError_t spec_launch_price(
    int32_t batch, int32_t K, int32_t L, const int32_t* d, const float* c, const int32_t* d_len,
    const int32_t* g, const int32_t* g_len, const int32_t* match_n, const int32_t* agree,
    const int32_t* copy_len, const spec_estimator* est, const float* table, float lambda,
    int32_t budget, int32_t mvl, int32_t policy, int32_t draft_greedy, int32_t* chain, float* S,
    int32_t* chain_len, int32_t* source, int32_t* verify_len, int32_t* row_off,
    uint8_t* point_mass, uint32_t* status, cudaStream_t stream) {
  spec::PriceParams p;
  p.batch = batch;
  p.K = K;
  p.L = L;
  p.d = d;
  p.c = c;
  p.d_len = d_len;
  p.g = g;
  p.g_len = g_len;
  p.match_n = match_n;
  p.agree = agree;
  p.copy_len = copy_len;
  p.table = table;
  p.tab_const = est->use_constant_h;
  p.n_full = est->n_full;
  p.m_cap = est->m_cap;
  p.lambda = lambda;
  p.budget = budget;
  p.mvl = mvl;
  p.policy = policy;
  p.draft_greedy = draft_greedy;
  p.chain = chain;
  p.S = S;
  p.chain_len = chain_len;
  p.source = source;
  p.verify_len = verify_len;
  p.row_off = row_off;
  p.point_mass = point_mass;
  p.status = status;
  int threads = ((batch + 31) / 32) * 32;
  if (threads < 32) threads = 32;
  const size_t smem = (size_t)L * (size_t)(batch > 0 ? batch : 1) * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(spec::price_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  spec::price_kernel<<<1, threads, smem, stream>>>(p);
  return cudaGetLastError();
}
