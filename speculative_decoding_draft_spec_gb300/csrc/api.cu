// api.cu -- the C ABI of include/spec.h: host-side argument validation,
// workspace layout, and the kernel launches of the four steps.  No entry point
// allocates device memory or synchronises with the host.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>
#include <math.h>

#include "common.cuh"

// pricing with the fixed scratch array (price.cu; internal, not exported)
__attribute__((visibility("hidden"))) cudaError_t spec_launch_price_static(
    int32_t batch, int32_t K, int32_t L, const int32_t* d, const float* c, const int32_t* d_len,
    const int32_t* g, const int32_t* g_len, const int32_t* match_n, const int32_t* agree,
    const int32_t* copy_len, const spec_estimator* est, const float* table, float lambda, int32_t budget,
    int32_t mvl, int32_t policy, int32_t draft_greedy, int32_t* chain, float* S, int32_t* chain_len,
    int32_t* source, int32_t* verify_len, int32_t* row_off, uint8_t* point_mass, uint32_t* status_word,
    cudaStream_t stream);

extern "C" {
cudaError_t spec_launch_ngram(const int32_t* hist, int64_t stride, const int32_t* hist_len,
                              int32_t batch, int32_t n_min, int32_t n_max, int32_t L, int32_t cap,
                              int32_t* g, int32_t* g_len, int32_t* match_n, int32_t* agree,
                              int32_t* copy_len, uint32_t* status, int num_sms, cudaStream_t stream,
                              int* unsupported);
size_t spec_estimator_entries(const spec_estimator* e, int32_t L);
cudaError_t spec_launch_estimator_table(const spec_estimator* e, int32_t L, float* table,
                                        cudaStream_t stream);
cudaError_t spec_launch_price(int32_t batch, int32_t K, int32_t L, const int32_t* d, const float* c,
                              const int32_t* d_len, const int32_t* g, const int32_t* g_len,
                              const int32_t* match_n, const int32_t* agree, const int32_t* copy_len,
                              const spec_estimator* est, const float* table, float lambda,
                              int32_t budget, int32_t mvl, int32_t policy, int32_t draft_greedy,
                              int32_t* chain, float* S, int32_t* chain_len, int32_t* source,
                              int32_t* verify_len, int32_t* row_off, uint8_t* point_mass,
                              uint32_t* status, uint32_t* keys, cudaStream_t stream);
cudaError_t spec_launch_build_tree(int32_t batch, int32_t P, int32_t Kc, const int32_t* anchor,
                                   const int32_t* cand_tok, const float* cand_score, const int32_t* ng_tok,
                                   int32_t n_chains, int32_t Lg, const int32_t* ng_len, const float* ng_score,
                                   const float* ng_adj,
                                   int32_t width, int32_t* tok, int32_t* parent, int32_t* cand_id,
                                   int32_t* n_rows, uint32_t* status, cudaStream_t stream);
cudaError_t spec_launch_ngram_fill(const int32_t* hist, int64_t hist_stride, const int32_t* hist_len,
                                   int32_t batch, int32_t P, int32_t Kc, const int32_t* cand_tok, int32_t n_min,
                                   int32_t copy_cap, int32_t max_depth, int32_t Lg, int32_t* ng_tok,
                                   int32_t* ng_len, int32_t* ng_ev, uint32_t* status, cudaStream_t stream);
cudaError_t spec_launch_size_budget(int32_t batch, int32_t L, const float* S, const int32_t* chain_len,
                                    int32_t mvl, double C0, double p, int32_t* out_budget, float* out_lambda,
                                    uint32_t* status, cudaStream_t stream);
cudaError_t spec_launch_sample_drafts(int32_t batch, int32_t K, int32_t vocab, int32_t dtype,
                                      const void* draft_logits, float temperature, uint64_t seed, uint64_t step,
                                      int32_t* y, float* dbg_u, float* dbg_q, const spec_workspace* ws,
                                      int num_sms, cudaStream_t stream);
cudaError_t spec_launch_draft_price(
    const int32_t* hist, int64_t stride, const int32_t* hist_len, int32_t batch, int32_t n_min, int32_t n_max,
    int32_t cap, int32_t* g, int32_t* g_len, int32_t* match_n, int32_t* agree, int32_t* copy_len, int32_t K,
    int32_t L, const int32_t* d, const float* c, const int32_t* d_len, const spec_estimator* est,
    const float* table, float lambda, int32_t budget, int32_t mvl, int32_t policy, int32_t draft_greedy,
    int32_t* chain, float* S, int32_t* chain_len, int32_t* source, int32_t* verify_len, int32_t* row_off,
    uint8_t* point_mass, uint32_t* status, uint32_t* keys, cudaStream_t stream, int* unsupported);
cudaError_t spec_launch_verify_chain(int32_t batch, int32_t vocab, int32_t dtype, const void* logits,
                                     const int32_t* row_off, const void* draft, int32_t K,
                                     const int32_t* chain, int32_t L, const int32_t* verify_len,
                                     const uint8_t* pm, float temperature, uint64_t seed,
                                     uint64_t step, int32_t* out_tokens, int32_t* n_accepted,
                                     int32_t* n_emitted, float* dbg_ratio, float* dbg_u,
                                     float* dbg_resid, int32_t q_reuse_base, const spec_workspace* ws,
                                     int num_sms, cudaStream_t stream);
int spec_verify_limits_ok(int32_t vocab, int32_t dtype, int64_t rows, int num_sms);
cudaError_t spec_launch_verify_tree(int32_t batch, int32_t vocab, int32_t dtype, const void* logits,
                                    const int32_t* node_off, const int32_t* tok,
                                    const int32_t* parent, int32_t max_nodes, int32_t* path,
                                    int32_t* accept_len, int32_t* out_tokens,
                                    const spec_workspace* ws, int num_sms, cudaStream_t stream);
}

namespace {

constexpr int32_t kMaxVerifyBatch = 2048;

int device_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  static int cached_dev = -1, cached = 0;
  if (dev != cached_dev) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cached = n;
    cached_dev = dev;
  }
  return cached;
}

spec_status from_cuda(cudaError_t e) { return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA; }

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

bool layout(int32_t max_batch, int32_t max_rows, int32_t K, int32_t vocab, spec_workspace* w) {
  if (max_batch < 0 || max_rows < 0 || K < 0 || vocab < 1 || K > SPEC_MAX_L || vocab > SPEC_MAX_VOCAB) return false;
  const int64_t units = ((int64_t)vocab + SPEC_UNIT - 1) / SPEC_UNIT;
  size_t off = 256;  // status word + padding
  w->off_counter = off;
  off = align256(off + sizeof(uint32_t) * (size_t)max_batch);
  w->off_counter2 = off;
  off = align256(off + sizeof(uint32_t) * (size_t)max_batch);
  w->off_record = off;
  off = align256(off + 64 * (size_t)max_batch);
  w->off_rowkey = off;
  off = align256(off + sizeof(unsigned long long) * (size_t)max_rows);
  const size_t pstride = (size_t)spec_partial_stride((int)units);
  w->off_partial = off;
  off = align256(off + sizeof(float2) * pstride * ((size_t)max_rows + (size_t)max_batch * K));
  w->off_partial2 = off;
  off = align256(off + sizeof(float) * pstride * (size_t)max_batch);
  w->off_keys = off;  // sized for the largest pricing batch, whatever max_batch is
  off = align256(off + sizeof(uint32_t) * (size_t)SPEC_MAX_PRICE_BATCH * SPEC_MAX_L);
  w->off_counter3 = off;
  off = align256(off + sizeof(uint32_t) * (size_t)max_batch * (size_t)(K > 1 ? K : 1));
  w->bytes = off;
  w->max_batch = max_batch;
  w->max_rows = max_rows;
  w->K = K;
  w->vocab = vocab;
  w->units = (int32_t)units;
  w->pad_ = 0;
  return true;
}

bool ws_ok(const spec_workspace* ws) {
  return ws && ws->base && (reinterpret_cast<uintptr_t>(ws->base) & 255u) == 0 &&
         ws->off_keys % 256 == 0 &&
         ws->bytes >= ws->off_keys + sizeof(uint32_t) * (size_t)SPEC_MAX_PRICE_BATCH * SPEC_MAX_L;
}

uint32_t* status_of(const spec_workspace* ws) { return static_cast<uint32_t*>(ws->base); }

uint32_t* keys_of(const spec_workspace* ws) {
  return reinterpret_cast<uint32_t*>(static_cast<char*>(ws->base) + ws->off_keys);
}

}  // namespace

extern "C" {

const char* spec_status_string(spec_status s) {
  switch (s) {
    case SPEC_OK: return "ok";
    case SPEC_ERR_INVALID_ARG: return "invalid argument";
    case SPEC_ERR_CUDA: return "CUDA error";
    case SPEC_ERR_UNSUPPORTED: return "unsupported size";
    case SPEC_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
  }
  return "unknown status";
}

int32_t spec_version(void) { return 1; }

size_t spec_workspace_bytes(int32_t max_batch, int32_t max_rows, int32_t K, int32_t vocab) {
  spec_workspace w;
  if (!layout(max_batch, max_rows, K, vocab, &w)) return 0;
  return w.bytes;
}

spec_status spec_workspace_init(spec_workspace* ws, void* dev_mem, size_t bytes, int32_t max_batch,
                                int32_t max_rows, int32_t K, int32_t vocab, cudaStream_t stream) {
  if (!ws || !dev_mem) return SPEC_ERR_INVALID_ARG;
  spec_workspace w;
  memset(&w, 0, sizeof w);
  if (!layout(max_batch, max_rows, K, vocab, &w)) return SPEC_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(dev_mem) & 255u) != 0 || bytes < w.bytes) return SPEC_ERR_WORKSPACE;
  w.base = dev_mem;
  w.bytes = bytes;
  *ws = w;
  return from_cuda(cudaMemsetAsync(dev_mem, 0, bytes, stream));
}

uint32_t* spec_workspace_status_word(const spec_workspace* ws) {
  return ws ? static_cast<uint32_t*>(ws->base) : nullptr;
}

size_t spec_estimator_table_bytes(const spec_estimator* est, int32_t L) {
  if (!est || L < 1 || L > SPEC_MAX_L) return 0;
  if (!est->use_constant_h && (est->m_cap < 1 || est->m_cap > SPEC_MAX_COPY_CAP || est->m_ref < 1))
    return 0;
  return spec_estimator_entries(est, L) * sizeof(float);
}

spec_status spec_estimator_build(const spec_estimator* est, int32_t L, float* table,
                                 size_t table_bytes, cudaStream_t stream) {
  if (!est || !table) return SPEC_ERR_INVALID_ARG;
  const size_t need = spec_estimator_table_bytes(est, L);
  if (need == 0) return SPEC_ERR_INVALID_ARG;
  if (table_bytes < need || (reinterpret_cast<uintptr_t>(table) & 15u) != 0) return SPEC_ERR_INVALID_ARG;
  return from_cuda(spec_launch_estimator_table(est, L, table, stream));
}

spec_status spec_ngram_propose(const int32_t* hist, int64_t hist_stride, const int32_t* hist_len,
                               int32_t batch, int32_t n_min, int32_t n_max, int32_t max_propose,
                               int32_t copy_cap, int32_t* g, int32_t* g_len, int32_t* match_n,
                               int32_t* agree, int32_t* copy_len, const spec_workspace* ws,
                               cudaStream_t stream) {
  if (batch < 0 || hist_stride < 0) return SPEC_ERR_INVALID_ARG;
  if (n_min < 1 || n_max < n_min || max_propose < 0 || copy_cap < n_max) return SPEC_ERR_INVALID_ARG;
  if (n_max > SPEC_MAX_N || max_propose > SPEC_MAX_L || copy_cap > SPEC_MAX_COPY_CAP)
    return SPEC_ERR_UNSUPPORTED;
  if (batch > 0 && (!hist_len || !g_len || !match_n || !agree || !copy_len ||
                    (max_propose > 0 && !g) || (hist_stride > 0 && !hist)))
    return SPEC_ERR_INVALID_ARG;
  if (!ws_ok(ws)) return SPEC_ERR_WORKSPACE;
  if (batch == 0) return SPEC_OK;
  const int sms = device_sms();
  if (sms <= 0) return SPEC_ERR_CUDA;
  int unsupported = 0;
  const cudaError_t e = spec_launch_ngram(hist, hist_stride < 1 ? 1 : hist_stride, hist_len, batch,
                                          n_min, n_max, max_propose, copy_cap, g, g_len, match_n,
                                          agree, copy_len, status_of(ws), sms, stream, &unsupported);
  if (unsupported) return SPEC_ERR_UNSUPPORTED;
  return from_cuda(e);
}

spec_status spec_price_and_allocate(
    int32_t batch, int32_t K, int32_t L, const int32_t* d, const float* c, const int32_t* d_len,
    const int32_t* g, const int32_t* g_len, const int32_t* match_n, const int32_t* agree,
    const int32_t* copy_len, const spec_estimator* est, const float* est_table,
    size_t est_table_bytes, float lambda, int32_t budget, int32_t max_verify_len, spec_policy policy,
    int32_t draft_greedy, int32_t* chain, float* S, int32_t* chain_len, int32_t* source,
    int32_t* verify_len, int32_t* row_off, uint8_t* point_mass, const spec_workspace* ws,
    cudaStream_t stream) {
  if (batch < 0 || K < 0 || L < 1 || K > L || budget < 0 || max_verify_len < 0 || !est ||
      !(lambda == lambda) || (int)policy < 0 || (int)policy > 4)
    return SPEC_ERR_INVALID_ARG;
  if (L > SPEC_MAX_L || batch > SPEC_MAX_PRICE_BATCH) return SPEC_ERR_UNSUPPORTED;
  if (!est_table || !row_off) return SPEC_ERR_INVALID_ARG;
  if (batch > 0 && (!d_len || !g || !g_len || !match_n || !agree || !copy_len || !chain || !S ||
                    !chain_len || !source || !verify_len || !point_mass || (K > 0 && (!d || !c))))
    return SPEC_ERR_INVALID_ARG;
  if (!est->use_constant_h && (est->m_cap < 1 || est->m_cap > SPEC_MAX_COPY_CAP)) return SPEC_ERR_INVALID_ARG;
  const size_t need = spec_estimator_table_bytes(est, L);
  if (need == 0 || est_table_bytes < need) return SPEC_ERR_INVALID_ARG;
  if (!ws_ok(ws)) return SPEC_ERR_WORKSPACE;
  return from_cuda(spec_launch_price(batch, K, L, d, c, d_len, g, g_len, match_n, agree, copy_len,
                                     est, est_table, lambda, budget, max_verify_len, (int32_t)policy,
                                     draft_greedy ? 1 : 0, chain, S, chain_len, source, verify_len,
                                     row_off, point_mass, status_of(ws), keys_of(ws), stream));
}

spec_status spec_price_and_allocate_static(
    int32_t batch, int32_t K, int32_t L, const int32_t* d, const float* c, const int32_t* d_len,
    const int32_t* g, const int32_t* g_len, const int32_t* match_n, const int32_t* agree,
    const int32_t* copy_len, const spec_estimator* est, const float* est_table,
    size_t est_table_bytes, float lambda, int32_t budget, int32_t max_verify_len, spec_policy policy,
    int32_t draft_greedy, int32_t* chain, float* S, int32_t* chain_len, int32_t* source,
    int32_t* verify_len, int32_t* row_off, uint8_t* point_mass, uint32_t* status_word,
    cudaStream_t stream) {
  // the checks of spec_price_and_allocate, then the fixed scratch's batch limit
  if (batch < 0 || K < 0 || L < 1 || K > L || budget < 0 || max_verify_len < 0 || !est ||
      !(lambda == lambda) || (int)policy < 0 || (int)policy > 4)
    return SPEC_ERR_INVALID_ARG;
  if (L > SPEC_MAX_L || batch > SPEC_STATIC_PRICE_MAX_BATCH) return SPEC_ERR_UNSUPPORTED;
  if (!est_table || !row_off) return SPEC_ERR_INVALID_ARG;
  if (batch > 0 && (!d_len || !g || !g_len || !match_n || !agree || !copy_len || !chain || !S ||
                    !chain_len || !source || !verify_len || !point_mass || (K > 0 && (!d || !c))))
    return SPEC_ERR_INVALID_ARG;
  if (!est->use_constant_h && (est->m_cap < 1 || est->m_cap > SPEC_MAX_COPY_CAP)) return SPEC_ERR_INVALID_ARG;
  const size_t need = spec_estimator_table_bytes(est, L);
  if (need == 0 || est_table_bytes < need) return SPEC_ERR_INVALID_ARG;
  return from_cuda(spec_launch_price_static(batch, K, L, d, c, d_len, g, g_len, match_n, agree, copy_len, est,
                                            est_table, lambda, budget, max_verify_len, (int32_t)policy,
                                            draft_greedy ? 1 : 0, chain, S, chain_len, source, verify_len,
                                            row_off, point_mass, status_word, stream));
}

spec_status spec_build_tree(int32_t batch, int32_t P, int32_t Kc, const int32_t* anchor,
                            const int32_t* cand_tok, const float* cand_score, const int32_t* ng_tok,
                            int32_t n_chains, int32_t Lg, const int32_t* ng_len, const float* ng_score,
                            const float* ng_adj, int32_t width, int32_t* tok, int32_t* parent, int32_t* cand_id,
                            int32_t* n_rows, const spec_workspace* ws, cudaStream_t stream) {
  if (batch < 0 || P < 0 || Kc < 1 || Lg < 0 || width < 1 || n_chains < 1 || n_chains > P + 1)
    return SPEC_ERR_INVALID_ARG;
  if ((int64_t)1 + (int64_t)P * Kc + (int64_t)n_chains * Lg > SPEC_MAX_TREE_CANDIDATES ||
      width > SPEC_MAX_TREE_NODES)
    return SPEC_ERR_UNSUPPORTED;
  if (batch > 0 && (!anchor || !ng_len || !ng_score || !ng_adj || !tok || !parent || !cand_id || !n_rows ||
                    (P > 0 && (!cand_tok || !cand_score)) || (Lg > 0 && !ng_tok)))
    return SPEC_ERR_INVALID_ARG;
  if (!ws_ok(ws)) return SPEC_ERR_WORKSPACE;
  if (batch == 0) return SPEC_OK;
  return from_cuda(spec_launch_build_tree(batch, P, Kc, anchor, cand_tok, cand_score, ng_tok, n_chains, Lg, ng_len,
                                          ng_score, ng_adj, width, tok, parent, cand_id, n_rows, status_of(ws),
                                          stream));
}

spec_status spec_ngram_fill(const int32_t* hist, int64_t hist_stride, const int32_t* hist_len, int32_t batch,
                            int32_t P, int32_t Kc, const int32_t* cand_tok, int32_t n_min, int32_t copy_cap,
                            int32_t max_depth, int32_t Lg, int32_t* ng_tok, int32_t* ng_len, int32_t* ng_ev,
                            const spec_workspace* ws, cudaStream_t stream) {
  if (batch < 0 || hist_stride < 0 || P < 0 || Kc < 1 || n_min < 1 || copy_cap < n_min || max_depth < 0 ||
      Lg < 0)
    return SPEC_ERR_INVALID_ARG;
  if ((int64_t)P + Lg > 4096 || batch > 65535) return SPEC_ERR_UNSUPPORTED;
  if (batch > 0 && (!hist_len || !ng_len || (hist_stride > 0 && !hist) || (P > 0 && !cand_tok) ||
                    (Lg > 0 && (!ng_tok || !ng_ev))))
    return SPEC_ERR_INVALID_ARG;
  if (!ws_ok(ws)) return SPEC_ERR_WORKSPACE;
  if (batch == 0) return SPEC_OK;
  return from_cuda(spec_launch_ngram_fill(hist, hist_stride, hist_len, batch, P, Kc, cand_tok, n_min, copy_cap,
                                          max_depth, Lg, ng_tok, ng_len, ng_ev, status_of(ws), stream));
}

spec_status spec_size_budget(int32_t batch, int32_t L, const float* S, const int32_t* chain_len,
                             int32_t max_verify_len, double C0, double p, int32_t* out_budget,
                             float* out_lambda, const spec_workspace* ws, cudaStream_t stream) {
  if (batch < 0 || L < 1 || max_verify_len < 0 || !(C0 > 0.0) || !(p > 0.0) || !(C0 < INFINITY) ||
      !(p < INFINITY))
    return SPEC_ERR_INVALID_ARG;
  if (L > SPEC_MAX_L || batch > SPEC_MAX_PRICE_BATCH) return SPEC_ERR_UNSUPPORTED;
  if (!out_budget || !out_lambda || (batch > 0 && (!S || !chain_len))) return SPEC_ERR_INVALID_ARG;
  if (!ws_ok(ws)) return SPEC_ERR_WORKSPACE;
  return from_cuda(spec_launch_size_budget(batch, L, S, chain_len, max_verify_len, C0, p, out_budget, out_lambda,
                                           status_of(ws), stream));
}

spec_status spec_sample_drafts(int32_t batch, int32_t K, int32_t vocab, spec_dtype dtype,
                               const void* draft_logits, float temperature, uint64_t seed, uint64_t step,
                               int32_t* y, float* dbg_u, float* dbg_q, const spec_workspace* ws,
                               cudaStream_t stream) {
  if (batch < 0 || K < 1 || vocab < 1 || !(temperature > 0.0f) || !(temperature < INFINITY))
    return SPEC_ERR_INVALID_ARG;
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_INVALID_ARG;
  if (K > SPEC_MAX_L || batch > kMaxVerifyBatch) return SPEC_ERR_UNSUPPORTED;
  if (batch > 0 && (!draft_logits || !y)) return SPEC_ERR_INVALID_ARG;
  if (!ws_ok(ws)) return SPEC_ERR_WORKSPACE;
  if (batch > ws->max_batch || K > ws->K || vocab > ws->vocab) return SPEC_ERR_WORKSPACE;
  if (batch == 0) return SPEC_OK;
  const int sms = device_sms();
  if (sms <= 0) return SPEC_ERR_CUDA;
  if (!spec_verify_limits_ok(vocab, (int32_t)dtype, (int64_t)batch * K, sms)) return SPEC_ERR_UNSUPPORTED;
  return from_cuda(spec_launch_sample_drafts(batch, K, vocab, (int32_t)dtype, draft_logits, temperature, seed, step,
                                             y, dbg_u, dbg_q, ws, sms, stream));
}

spec_status spec_draft_and_price(
    const int32_t* hist, int64_t hist_stride, const int32_t* hist_len, int32_t batch, int32_t n_min,
    int32_t n_max, int32_t copy_cap, int32_t* g, int32_t* g_len, int32_t* match_n, int32_t* agree,
    int32_t* copy_len, int32_t K, int32_t L, const int32_t* d, const float* c, const int32_t* d_len,
    const spec_estimator* est, const float* est_table, size_t est_table_bytes, float lambda,
    int32_t budget, int32_t max_verify_len, spec_policy policy, int32_t draft_greedy, int32_t* chain,
    float* S, int32_t* chain_len, int32_t* source, int32_t* verify_len, int32_t* row_off,
    uint8_t* point_mass, const spec_workspace* ws, cudaStream_t stream) {
  // the checks of both steps
  if (batch < 0 || hist_stride < 0 || K < 0 || L < 1 || K > L || budget < 0 || max_verify_len < 0 || !est ||
      !(lambda == lambda) || (int)policy < 0 || (int)policy > 4)
    return SPEC_ERR_INVALID_ARG;
  if (n_min < 1 || n_max < n_min || copy_cap < n_max) return SPEC_ERR_INVALID_ARG;
  if (n_max > SPEC_MAX_N || L > SPEC_MAX_L || copy_cap > SPEC_MAX_COPY_CAP || batch > SPEC_MAX_PRICE_BATCH)
    return SPEC_ERR_UNSUPPORTED;
  if (!est_table || !row_off) return SPEC_ERR_INVALID_ARG;
  if (batch > 0 && (!hist_len || !g || !g_len || !match_n || !agree || !copy_len || !d_len || !chain || !S ||
                    !chain_len || !source || !verify_len || !point_mass || (K > 0 && (!d || !c)) ||
                    (hist_stride > 0 && !hist)))
    return SPEC_ERR_INVALID_ARG;
  if (!est->use_constant_h && (est->m_cap < 1 || est->m_cap > SPEC_MAX_COPY_CAP)) return SPEC_ERR_INVALID_ARG;
  const size_t need = spec_estimator_table_bytes(est, L);
  if (need == 0 || est_table_bytes < need) return SPEC_ERR_INVALID_ARG;
  if (!ws_ok(ws)) return SPEC_ERR_WORKSPACE;
  if (batch == 0) {
    // nothing to draft or price: an empty layout
    return from_cuda(cudaMemsetAsync(row_off, 0, sizeof(int32_t), stream));
  }
  int unsupported = 0;
  const cudaError_t e = spec_launch_draft_price(
      hist, hist_stride < 1 ? 1 : hist_stride, hist_len, batch, n_min, n_max, copy_cap, g, g_len, match_n, agree,
      copy_len, K, L, d, c, d_len, est, est_table, lambda, budget, max_verify_len, (int32_t)policy,
      draft_greedy ? 1 : 0, chain, S, chain_len, source, verify_len, row_off, point_mass, status_of(ws), keys_of(ws),
      stream, &unsupported);
  if (unsupported) return SPEC_ERR_UNSUPPORTED;
  return from_cuda(e);
}

}  // extern "C"

namespace {

// spec_verify_chain (reuse 0) and spec_verify_chain_drafted (reuse 1)
spec_status verify_chain(int32_t batch, int32_t vocab, spec_dtype dtype, const void* target_logits,
                         const int32_t* row_off, int32_t max_rows, const void* draft_logits, int32_t K,
                         const int32_t* chain, int32_t L, const int32_t* verify_len, const uint8_t* point_mass,
                         float temperature, uint64_t seed, uint64_t step, int32_t* out_tokens,
                         int32_t* n_accepted, int32_t* n_emitted, float* dbg_ratio, float* dbg_u,
                         float* dbg_resid, int reuse, const spec_workspace* ws, cudaStream_t stream) {
  if (batch < 0 || vocab < 1 || L < 1 || K < 0 || max_rows < 0 || !(temperature == temperature))
    return SPEC_ERR_INVALID_ARG;
  if (reuse && (!draft_logits || !point_mass || !(temperature > 0.0f))) return SPEC_ERR_INVALID_ARG;
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_INVALID_ARG;
  if (L > SPEC_MAX_L || K > SPEC_MAX_L || batch > kMaxVerifyBatch) return SPEC_ERR_UNSUPPORTED;
  if (!row_off) return SPEC_ERR_INVALID_ARG;
  if (batch > 0 && (!target_logits || !chain || !verify_len || !out_tokens || !n_accepted || !n_emitted))
    return SPEC_ERR_INVALID_ARG;
  if (draft_logits && K < 1) return SPEC_ERR_INVALID_ARG;
  if (!ws_ok(ws)) return SPEC_ERR_WORKSPACE;
  if (batch > ws->max_batch || max_rows > ws->max_rows || vocab > ws->vocab ||
      (draft_logits && K > ws->K))
    return SPEC_ERR_WORKSPACE;
  if (batch == 0) return SPEC_OK;
  const int sms = device_sms();
  if (sms <= 0) return SPEC_ERR_CUDA;
  if (!spec_verify_limits_ok(vocab, (int32_t)dtype, (int64_t)max_rows + (int64_t)batch * K, sms))
    return SPEC_ERR_UNSUPPORTED;
  spec_workspace w = *ws;
  w.max_rows = max_rows;  // the call's row bound; partial slots of draft rows follow it, except when
                          // they are reused: they sit where spec_sample_drafts put them, after the
                          // workspace's row capacity
  return from_cuda(spec_launch_verify_chain(batch, vocab, (int32_t)dtype, target_logits, row_off,
                                            draft_logits, K, chain, L, verify_len, point_mass,
                                            temperature, seed, step, out_tokens, n_accepted,
                                            n_emitted, dbg_ratio, dbg_u, dbg_resid, reuse ? ws->max_rows : -1,
                                            &w, sms, stream));
}

}  // namespace

extern "C" {

spec_status spec_verify_chain(int32_t batch, int32_t vocab, spec_dtype dtype, const void* target_logits,
                              const int32_t* row_off, int32_t max_rows, const void* draft_logits,
                              int32_t K, const int32_t* chain, int32_t L, const int32_t* verify_len,
                              const uint8_t* point_mass, float temperature, uint64_t seed,
                              uint64_t step, int32_t* out_tokens, int32_t* n_accepted,
                              int32_t* n_emitted, float* dbg_ratio, float* dbg_u, float* dbg_resid,
                              const spec_workspace* ws, cudaStream_t stream) {
  return verify_chain(batch, vocab, dtype, target_logits, row_off, max_rows, draft_logits, K, chain, L,
                      verify_len, point_mass, temperature, seed, step, out_tokens, n_accepted, n_emitted,
                      dbg_ratio, dbg_u, dbg_resid, 0, ws, stream);
}

spec_status spec_verify_chain_drafted(int32_t batch, int32_t vocab, spec_dtype dtype, const void* target_logits,
                                      const int32_t* row_off, int32_t max_rows, const void* draft_logits,
                                      int32_t K, const int32_t* chain, int32_t L, const int32_t* verify_len,
                                      const uint8_t* point_mass, float temperature, uint64_t seed,
                                      uint64_t step, int32_t* out_tokens, int32_t* n_accepted,
                                      int32_t* n_emitted, float* dbg_ratio, float* dbg_u, float* dbg_resid,
                                      const spec_workspace* ws, cudaStream_t stream) {
  return verify_chain(batch, vocab, dtype, target_logits, row_off, max_rows, draft_logits, K, chain, L,
                      verify_len, point_mass, temperature, seed, step, out_tokens, n_accepted, n_emitted,
                      dbg_ratio, dbg_u, dbg_resid, 1, ws, stream);
}

spec_status spec_verify_tree(int32_t batch, int32_t vocab, spec_dtype dtype, const void* logits,
                             const int32_t* node_off, int32_t max_rows, const int32_t* tok,
                             const int32_t* parent, int32_t max_nodes, int32_t* path,
                             int32_t* accept_len, int32_t* out_tokens, const spec_workspace* ws,
                             cudaStream_t stream) {
  if (batch < 0 || vocab < 1 || max_nodes < 1 || max_rows < 0) return SPEC_ERR_INVALID_ARG;
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_INVALID_ARG;
  if (max_nodes > SPEC_MAX_TREE_NODES || batch > kMaxVerifyBatch) return SPEC_ERR_UNSUPPORTED;
  if (!node_off) return SPEC_ERR_INVALID_ARG;
  if (batch > 0 && (!logits || !tok || !parent || !path || !accept_len || !out_tokens))
    return SPEC_ERR_INVALID_ARG;
  if (!ws_ok(ws)) return SPEC_ERR_WORKSPACE;
  if (batch > ws->max_batch || max_rows > ws->max_rows || vocab > ws->vocab) return SPEC_ERR_WORKSPACE;
  if (batch == 0) return SPEC_OK;
  const int sms = device_sms();
  if (sms <= 0) return SPEC_ERR_CUDA;
  if (!spec_verify_limits_ok(vocab, (int32_t)dtype, (int64_t)max_rows, sms)) return SPEC_ERR_UNSUPPORTED;
  spec_workspace w = *ws;
  w.max_rows = max_rows;
  return from_cuda(spec_launch_verify_tree(batch, vocab, (int32_t)dtype, logits, node_off, tok, parent,
                                           max_nodes, path, accept_len, out_tokens, &w, sms, stream));
}

}  // extern "C"
