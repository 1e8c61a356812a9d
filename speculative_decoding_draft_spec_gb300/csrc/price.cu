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
// GB300 layout, one launch: phase 1 gives every request one warp (lane k stages
// position k+1 of the request's rows in shared memory in one coalesced round
// trip; the survivals and chain values are then formed left to right, so the
// fp32 results equal the sequential definition bit for bit) and writes one
// allocation key per slot.  Phase 2 runs in the last CTA to arrive (an
// acquire-release counter, no waiting): the budget-th largest key is found by
// a four-pass radix select with per-warp shared-memory histograms, and one
// block scan of the per-request (above, tie) counts gives verify_len and the
// row offsets.
#include "pricing.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

namespace spec {

// ------------------------------------------------------------------ Eq. (1)
struct EstimatorDev {
  double beta[32];
  double w_first, w_rest, delta, ell_first, ell_rest, kappa_first, kappa_rest;
  int32_t n_ref, n_full, m_cap, m_ref, use_constant_h;
  double constant_h;
};

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
    // layout: part A [(n * 2 + a) * L + k-1], n in [0, 32], a in {0, 1};
    //         part B [(a * (m_cap + 1) + m) * L + k-1] for n = n_full
    // so one request's h_1..h_L are contiguous
    int32_t k, n, a, m;
    bool full;
    if (idx < partA) {
      k = (int32_t)(idx % L) + 1;
      const int32_t na = (int32_t)(idx / L);
      n = na / 2;
      a = na % 2;
      m = n;
      full = false;
    } else {
      const int64_t j = idx - partA;
      k = (int32_t)(j % L) + 1;
      const int32_t am = (int32_t)(j / L);
      a = am / (e.m_cap + 1);
      m = am % (e.m_cap + 1);
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
  int32_t batch;
  const int32_t* d;
  const float* c;
  const int32_t* d_len;
  const int32_t* g;
  const int32_t* g_len;
  const int32_t* match_n;
  const int32_t* agree;
  const int32_t* copy_len;
  PriceCtx cx;
  SelectCtx sc;
  uint32_t* status;
  uint32_t* arrive;  // CTA arrival counter (zero between calls)
};

#define PR_WARPS 8
#define PR_THREADS (32 * PR_WARPS)

// One warp per request; the last CTA to arrive (acquire-release counter, no
// waiting) allocates the budget for the whole batch with one warp.
__global__ void __launch_bounds__(PR_THREADS, 1) price_kernel(PriceParams p) {
  extern __shared__ __align__(16) int32_t s_scratch[];  // select_scratch_ints(batch, L)
  __shared__ PriceStage s_ps[PR_WARPS];
  __shared__ int32_t s_last;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  {
    uint32_t st = 0;
    const int r = blockIdx.x * PR_WARPS + warp;
    if (r < p.batch) {
      const int32_t K = p.cx.K, L = p.cx.L;
      const int32_t gl = p.g_len[r], n = p.match_n[r], a = p.agree[r], m = p.copy_len[r], dl = p.d_len[r];
      PriceStage& ps = s_ps[warp];
      if (lane < L) ps.g[lane] = p.g[(int64_t)r * L + lane];
      if (lane < K) {
        ps.d[lane] = p.d[(int64_t)r * K + lane];
        ps.c[lane] = p.c[(int64_t)r * K + lane];
      }
      __syncwarp();
      price_request_warp(p.cx, r, lane, ps, gl, n, a, m, dl, st, nullptr);
    }
    if (st) set_status(p.status, st);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint32_t old = atomic_add_acq_rel(p.arrive, 1u);
    s_last = (old + 1u == gridDim.x);
    if (s_last) *p.arrive = 0u;  // ready for the next call
  }
  __syncthreads();
  if (!s_last) return;
  select_budget_cta(p.sc, s_scratch);
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
    uint8_t* point_mass, uint32_t* status, uint32_t* keys, cudaStream_t stream) {
  spec::PriceParams p;
  p.batch = batch;
  p.d = d;
  p.c = c;
  p.d_len = d_len;
  p.g = g;
  p.g_len = g_len;
  p.match_n = match_n;
  p.agree = agree;
  p.copy_len = copy_len;
  p.cx.K = K;
  p.cx.L = L;
  p.cx.table = table;
  p.cx.tab_const = est->use_constant_h;
  p.cx.n_full = est->n_full;
  p.cx.m_cap = est->m_cap;
  p.cx.lambda = lambda;
  p.cx.policy = policy;
  p.cx.draft_greedy = draft_greedy;
  p.cx.chain = chain;
  p.cx.S = S;
  p.cx.chain_len = chain_len;
  p.cx.source = source;
  p.cx.point_mass = point_mass;
  p.cx.mvl = mvl;
  p.cx.keys = keys;
  p.sc.batch = batch;
  p.sc.L = L;
  p.sc.budget = budget;
  p.sc.keys = keys;
  p.sc.verify_len = verify_len;
  p.sc.row_off = row_off;
  p.status = status;
  p.arrive = status + 1;  // the word after the status word in the workspace header
  const int blocks = batch > 0 ? (batch + PR_WARPS - 1) / PR_WARPS : 1;
  const size_t smem = (size_t)spec::select_scratch_ints(batch > 0 ? batch : 1, L) * sizeof(int32_t);
  cudaError_t e = cudaFuncSetAttribute(spec::price_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  spec::price_kernel<<<blocks, PR_THREADS, smem, stream>>>(p);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Pricing without a workspace: the scratch of one call (status word, arrival
// counter, allocation keys) lives in a fixed array of this library's device
// memory, so neither the call nor its kernel allocates.  For callers that own
// no device workspace; calls that may overlap on one device race on the array.
// ---------------------------------------------------------------------------
namespace spec {
constexpr int kStaticHeaderWords = 64;  // [0] status word, [1] arrival counter
static __device__ __align__(256) uint32_t
    g_static_price_scratch[kStaticHeaderWords + SPEC_STATIC_PRICE_MAX_BATCH * SPEC_MAX_L];
}  // namespace spec

namespace {
constexpr int kMaxDevices = 256;
std::mutex g_static_mu;
// per device: the id of the context the address was looked up in, and the address
struct StaticAddr {
  unsigned long long ctx_id;
  uint32_t* addr;
};
StaticAddr g_static_addr[kMaxDevices] = {};
PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;
bool g_ctx_fns = false;

// Process-unique id of the calling thread's current context (the driver never
// hands an id out twice in one process, unlike a context handle, whose value
// can come back after the context is destroyed); 0 when there is none.
unsigned long long current_context_id() {
  if (!g_ctx_fns) {
    g_ctx_fns = true;
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f);
  }
  if (!g_ctx_current || !g_ctx_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (g_ctx_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  if (g_ctx_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}
}  // namespace

// Device address of the fixed scratch array in the current device's current
// context.  It is looked up (cudaGetSymbolAddress, with that device current)
// the first time a context calls, and kept with the context's id: a call from
// another context -- after cudaDeviceReset, or from a driver-API context on the
// same device -- looks it up again, so no address outlives its context.
// (Internal: not exported from the library.)
__attribute__((visibility("hidden"))) cudaError_t spec_static_price_scratch(uint32_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_static_mu);
  const unsigned long long id = current_context_id();
  StaticAddr& slot = g_static_addr[dev];
  if (id != 0 && slot.addr != nullptr && slot.ctx_id == id) {
    *out = slot.addr;
    return cudaSuccess;
  }
  void* addr = nullptr;
  e = cudaGetSymbolAddress(&addr, spec::g_static_price_scratch);
  if (e != cudaSuccess) return e;
  // the lookup makes the device's primary context current when none was
  slot.ctx_id = id != 0 ? id : current_context_id();
  slot.addr = static_cast<uint32_t*>(addr);
  *out = slot.addr;
  return cudaSuccess;
}

__attribute__((visibility("hidden"))) cudaError_t spec_launch_price_static(
    int32_t batch, int32_t K, int32_t L, const int32_t* d, const float* c, const int32_t* d_len,
    const int32_t* g, const int32_t* g_len, const int32_t* match_n, const int32_t* agree,
    const int32_t* copy_len, const spec_estimator* est, const float* table, float lambda,
    int32_t budget, int32_t mvl, int32_t policy, int32_t draft_greedy, int32_t* chain, float* S,
    int32_t* chain_len, int32_t* source, int32_t* verify_len, int32_t* row_off,
    uint8_t* point_mass, uint32_t* status_word, cudaStream_t stream) {
  if (batch > SPEC_STATIC_PRICE_MAX_BATCH || L > SPEC_MAX_L) return cudaErrorInvalidValue;
  uint32_t* scratch = nullptr;
  cudaError_t e = spec_static_price_scratch(&scratch);
  if (e != cudaSuccess) return e;
  uint32_t* keys = scratch + spec::kStaticHeaderWords;
  spec::PriceParams p;
  p.batch = batch;
  p.d = d;
  p.c = c;
  p.d_len = d_len;
  p.g = g;
  p.g_len = g_len;
  p.match_n = match_n;
  p.agree = agree;
  p.copy_len = copy_len;
  p.cx.K = K;
  p.cx.L = L;
  p.cx.table = table;
  p.cx.tab_const = est->use_constant_h;
  p.cx.n_full = est->n_full;
  p.cx.m_cap = est->m_cap;
  p.cx.lambda = lambda;
  p.cx.policy = policy;
  p.cx.draft_greedy = draft_greedy;
  p.cx.chain = chain;
  p.cx.S = S;
  p.cx.chain_len = chain_len;
  p.cx.source = source;
  p.cx.point_mass = point_mass;
  p.cx.mvl = mvl;
  p.cx.keys = keys;
  p.sc.batch = batch;
  p.sc.L = L;
  p.sc.budget = budget;
  p.sc.keys = keys;
  p.sc.verify_len = verify_len;
  p.sc.row_off = row_off;
  p.status = status_word ? status_word : scratch;  // scratch[0]: a word nobody reads
  p.arrive = scratch + 1;
  const int blocks = batch > 0 ? (batch + PR_WARPS - 1) / PR_WARPS : 1;
  const size_t smem = (size_t)spec::select_scratch_ints(batch > 0 ? batch : 1, L) * sizeof(int32_t);
  e = cudaFuncSetAttribute(spec::price_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  spec::price_kernel<<<blocks, PR_THREADS, smem, stream>>>(p);
  return cudaGetLastError();
}
