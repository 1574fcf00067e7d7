// C ABI of the draft-tree hot path: host-side argument checks and launches.
// Every function validates its arguments before any CUDA call and returns a
// negative BASTION_ERR_* code without launching when a check fails.
#include <cuda_runtime.h>
#include <stdint.h>

#include "bastion.h"

namespace bastion {
size_t topk_workspace_bytes(int B, int b, int V, int K, int es);
int topk_max_smem_ok(int V, int K, int es);
int launch_topk(const void *logits, int dtype, int B, int b, int V, int64_t ld, int K,
                float *topk_logq, float *topk_logit, int32_t *topk_tok, double *lse, void *ws,
                int32_t *status, cudaStream_t stream);
size_t lm_head_workspace_bytes(int rows, int V, int K);
int launch_lm_head(const void *hidden, const void *weight, int B, int b, int H, int V, int K,
                   float *topk_logq, float *topk_logit, int32_t *topk_tok, double *lse, void *ws,
                   int32_t *status, cudaStream_t stream);
int launch_build_tree(const float *topk_logit, const int32_t *topk_tok, const double *lse, int B,
                      int b, int K, int n_max, const int32_t *root_token, const int32_t *ctx_len,
                      const float *cost_ms, int cost_per_request, const float *l_ar,
                      int32_t *n_nodes, int32_t *parent, int32_t *depth, int32_t *pos_id,
                      int32_t *token, int32_t *rank, float *log_rho, float *a_hat, float *speedup,
                      uint32_t *anc_mask, int32_t *status, cudaStream_t stream);
size_t verify_workspace_bytes(int B, int n_max);
size_t mixture_tree_smem_bytes(int Z, int b, int K, int n_max);
size_t mixture_tree_ws_stride(int Z, int b, int K, int n_max);
int launch_build_tree_mixture(const float *topk_logit, const int32_t *topk_tok, const double *lse,
                              const double *pi, int B, int Z, int b, int K, int n_max,
                              const int32_t *root_token, const int32_t *ctx_len,
                              const float *cost_ms, int cost_per_request, const float *l_ar,
                              int32_t *n_nodes, int32_t *parent, int32_t *depth, int32_t *pos_id,
                              int32_t *token, float *log_rho, float *a_hat, float *speedup,
                              uint32_t *anc_mask, void *workspace, int32_t *status,
                              cudaStream_t stream);
int launch_verify(const void *target, int dtype, int B, int n_max, int V, int64_t ld, int b,
                  const int32_t *n_nodes, const int32_t *parent, const int32_t *token,
                  int32_t *argmax, int32_t *accept_len, int32_t *accept_nodes,
                  int32_t *out_tokens, void *ws, int32_t *status, cudaStream_t stream);
size_t verify_sample_workspace_bytes(int B, int n_max, int V);
int launch_verify_sample(const void *target, int dtype, int B, int n_max, int V, int64_t ld, int b,
                         float temperature, const double *uniforms, const int32_t *n_nodes,
                         const int32_t *parent, const int32_t *token, int32_t *sampled,
                         int32_t *accept_len, int32_t *accept_nodes, int32_t *out_tokens, void *ws,
                         int32_t *status, cudaStream_t stream);
int launch_calibrate(const float *sample_n, const float *sample_ms, int n_samples, double bytes0,
                     double bytes1, double flops0, double flops1, double bw, double peak,
                     double t_draft, int n_max, float *cost_ms, float *params, int32_t *status,
                     cudaStream_t stream);
size_t attention_workspace_bytes(int B, int n_max, int Hq, int Hkv, int D, int64_t L_cap);
int launch_attention(const void *q, const void *k, const void *v, int B, int n_max, int Hq,
                     int Hkv, int D, int64_t L_cap, const int32_t *ctx_len,
                     const int32_t *n_nodes, const uint32_t *anc_mask, float scale, void *out,
                     void *ws, int32_t *status, cudaStream_t stream);
}  // namespace bastion

namespace {

bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

}  // namespace

extern "C" {

const char *bastion_version(void) { return "bastion-gb300 0.1.0 sm_103a"; }

const char *bastion_status_string(int code) {
  switch (code) {
    case BASTION_OK: return "ok";
    case BASTION_ERR_NULL: return "a required pointer is null";
    case BASTION_ERR_SIZE: return "a size, count or stride is out of range";
    case BASTION_ERR_DTYPE: return "unknown dtype";
    case BASTION_ERR_ALIGN: return "a pointer misses its documented alignment";
    case BASTION_ERR_WORKSPACE: return "workspace missing or too small";
    case BASTION_ERR_UNSUPPORTED: return "valid arguments that the library does not support";
    case BASTION_ERR_LAUNCH: return "the CUDA launch reported an error";
    case BASTION_STATUS_NONFINITE: return "a NaN or +inf logit";
    case BASTION_STATUS_EMPTY_ROW: return "a drafter row with no finite logit";
    case BASTION_STATUS_BAD_COST: return "a cost C(N) that is not positive and finite";
    case BASTION_STATUS_KV_OVERFLOW: return "ctx_len + n_nodes exceeds the KV cache capacity";
    case BASTION_STATUS_BAD_TREE: return "n_nodes outside [1, n_max]";
    case BASTION_STATUS_BAD_WEIGHT: return "a mixture weight is negative or not finite";
    case BASTION_STATUS_TIMEOUT: return "a bounded device wait ran out";
    default: return "unknown code";
  }
}

size_t bastion_topk_marginals_workspace_bytes(int B, int b, int V, int K) {
  if (B < 1 || b < 1 || b > 32 || V < 1 || K < 1 || K > 1024 || K > V) return 0;
  size_t w2 = bastion::topk_workspace_bytes(B, b, V, K, 2);
  size_t w4 = bastion::topk_workspace_bytes(B, b, V, K, 4);
  return w2 > w4 ? w2 : w4;
}

int bastion_topk_marginals(const void *logits, int dtype, int B, int b, int V, int64_t ld_row,
                           int K, float *topk_logq, float *topk_logit, int32_t *topk_tok,
                           double *lse, void *workspace, size_t workspace_bytes,
                           int32_t *status, bastion_stream_t stream) {
  if (!logits || !topk_logit || !topk_tok || !lse || !status || !workspace) return BASTION_ERR_NULL;
  if (dtype != BASTION_F32 && dtype != BASTION_BF16) return BASTION_ERR_DTYPE;
  if (B < 1 || b < 1 || b > 32 || V < 1 || V >= (1 << 30) || K < 1 || K > 1024 || K > V ||
      ld_row < V)
    return BASTION_ERR_SIZE;
  const int es = dtype == BASTION_F32 ? 4 : 2;
  if (!aligned(logits, es) || !aligned(workspace, 256)) return BASTION_ERR_ALIGN;
  if (workspace_bytes < bastion::topk_workspace_bytes(B, b, V, K, es)) return BASTION_ERR_WORKSPACE;
  if (!bastion::topk_max_smem_ok(V, K, es)) return BASTION_ERR_UNSUPPORTED;
  if ((long long)B * b > (1LL << 24)) return BASTION_ERR_SIZE;
  return bastion::launch_topk(logits, dtype, B, b, V, ld_row, K, topk_logq, topk_logit, topk_tok,
                              lse, workspace, status, (cudaStream_t)stream);
}

size_t bastion_lm_head_topk_workspace_bytes(int B, int b, int V, int K) {
  if (B < 1 || b < 1 || (long long)B * b > (1LL << 24) || V < 1 || K < 1 || K > 64 || K > V) return 0;
  return bastion::lm_head_workspace_bytes(B * b, V, K);
}

int bastion_lm_head_topk(const void *hidden, const void *weight, int B, int b, int H, int V, int K,
                         float *topk_logq, float *topk_logit, int32_t *topk_tok, double *lse,
                         void *workspace, size_t workspace_bytes, int32_t *status,
                         bastion_stream_t stream) {
  if (!hidden || !weight || !topk_logit || !topk_tok || !lse || !status || !workspace)
    return BASTION_ERR_NULL;
  if (B < 1 || b < 1 || (long long)B * b > (1LL << 24) || V < 1 || K < 1 || K > 64 || K > V ||
      H < 1 || H > (1 << 20))
    return BASTION_ERR_SIZE;
  if (H % 64) return BASTION_ERR_UNSUPPORTED;
  if (!aligned(hidden, 16) || !aligned(weight, 16) || !aligned(workspace, 256) || !aligned(lse, 8))
    return BASTION_ERR_ALIGN;
  if (workspace_bytes < bastion_lm_head_topk_workspace_bytes(B, b, V, K)) return BASTION_ERR_WORKSPACE;
  return bastion::launch_lm_head(hidden, weight, B, b, H, V, K, topk_logq, topk_logit, topk_tok, lse,
                                 workspace, status, (cudaStream_t)stream);
}

int bastion_build_tree(const float *topk_logit, const int32_t *topk_tok, const double *lse,
                       int B, int b, int K, int n_max, const int32_t *root_token,
                       const int32_t *ctx_len, const float *cost_ms, int cost_per_request,
                       const float *l_ar, int32_t *n_nodes, int32_t *parent, int32_t *depth,
                       int32_t *pos_id, int32_t *token, int32_t *rank, float *log_rho,
                       float *a_hat, float *speedup, uint32_t *anc_mask, int32_t *status,
                       bastion_stream_t stream) {
  if (!topk_logit || !topk_tok || !lse || !root_token || !ctx_len || !cost_ms || !l_ar ||
      !n_nodes || !parent || !depth || !pos_id || !token || !rank || !log_rho || !a_hat ||
      !speedup || !anc_mask || !status)
    return BASTION_ERR_NULL;
  if (B < 1 || B > (1 << 24) || b < 1 || b > 32 || K < 1 || K > 1024 || n_max < 1 || n_max > 256)
    return BASTION_ERR_SIZE;
  if (!aligned(lse, 8)) return BASTION_ERR_ALIGN;
  return bastion::launch_build_tree(topk_logit, topk_tok, lse, B, b, K, n_max, root_token,
                                    ctx_len, cost_ms, cost_per_request, l_ar, n_nodes, parent,
                                    depth, pos_id, token, rank, log_rho, a_hat, speedup, anc_mask,
                                    status, (cudaStream_t)stream);
}

static bool mixture_sizes_ok(int B, int Z, int b, int K, int n_max) {
  return !(B < 1 || B > (1 << 24) || Z < 1 || Z > 32 || b < 1 || b > 32 || K < 1 || K > 1024 ||
           n_max < 1 || n_max > 256);
}

size_t bastion_build_tree_mixture_workspace_bytes(int B, int Z, int b, int K, int n_max) {
  if (!mixture_sizes_ok(B, Z, b, K, n_max)) return 0;
  return (size_t)B * bastion::mixture_tree_ws_stride(Z, b, K, n_max);
}

int bastion_build_tree_mixture(const float *topk_logit, const int32_t *topk_tok, const double *lse,
                               const double *pi, int B, int Z, int b, int K, int n_max,
                               const int32_t *root_token, const int32_t *ctx_len,
                               const float *cost_ms, int cost_per_request, const float *l_ar,
                               int32_t *n_nodes, int32_t *parent, int32_t *depth, int32_t *pos_id,
                               int32_t *token, float *log_rho, float *a_hat, float *speedup,
                               uint32_t *anc_mask, void *workspace, size_t workspace_bytes,
                               int32_t *status, bastion_stream_t stream) {
  if (!topk_logit || !topk_tok || !lse || !pi || !root_token || !ctx_len || !cost_ms || !l_ar ||
      !n_nodes || !parent || !depth || !pos_id || !token || !log_rho || !a_hat || !speedup ||
      !anc_mask || !workspace || !status)
    return BASTION_ERR_NULL;
  if (!mixture_sizes_ok(B, Z, b, K, n_max)) return BASTION_ERR_SIZE;
  if (!aligned(lse, 8) || !aligned(pi, 8) || !aligned(workspace, 256)) return BASTION_ERR_ALIGN;
  if (workspace_bytes < (size_t)B * bastion::mixture_tree_ws_stride(Z, b, K, n_max))
    return BASTION_ERR_WORKSPACE;
  if (bastion::mixture_tree_smem_bytes(Z, b, K, n_max) > (size_t)227 * 1024) return BASTION_ERR_UNSUPPORTED;
  return bastion::launch_build_tree_mixture(topk_logit, topk_tok, lse, pi, B, Z, b, K, n_max,
                                            root_token, ctx_len, cost_ms, cost_per_request, l_ar,
                                            n_nodes, parent, depth, pos_id, token, log_rho, a_hat,
                                            speedup, anc_mask, workspace, status,
                                            (cudaStream_t)stream);
}

size_t bastion_verify_greedy_workspace_bytes(int B, int n_max, int V) {
  if (B < 1 || B > 4096 || n_max < 1 || n_max > 256 || V < 1) return 0;
  return bastion::verify_workspace_bytes(B, n_max);
}

int bastion_verify_greedy(const void *target_logits, int dtype, int B, int n_max, int V,
                          int64_t ld_row, int b, const int32_t *n_nodes, const int32_t *parent,
                          const int32_t *token, int32_t *argmax, int32_t *accept_len,
                          int32_t *accept_nodes, int32_t *out_tokens, void *workspace,
                          size_t workspace_bytes, int32_t *status, bastion_stream_t stream) {
  if (!target_logits || !n_nodes || !parent || !token || !argmax || !accept_len ||
      !accept_nodes || !out_tokens || !workspace || !status)
    return BASTION_ERR_NULL;
  if (dtype != BASTION_F32 && dtype != BASTION_BF16) return BASTION_ERR_DTYPE;
  if (B < 1 || B > 4096 || n_max < 1 || n_max > 256 || V < 1 || V >= (1 << 30) || ld_row < V ||
      b < 1 || b > 32)
    return BASTION_ERR_SIZE;
  const int es = dtype == BASTION_F32 ? 4 : 2;
  if (!aligned(target_logits, es) || !aligned(workspace, 256)) return BASTION_ERR_ALIGN;
  if (workspace_bytes < bastion::verify_workspace_bytes(B, n_max)) return BASTION_ERR_WORKSPACE;
  return bastion::launch_verify(target_logits, dtype, B, n_max, V, ld_row, b, n_nodes, parent,
                                token, argmax, accept_len, accept_nodes, out_tokens, workspace,
                                status, (cudaStream_t)stream);
}

size_t bastion_verify_sample_workspace_bytes(int B, int n_max, int V) {
  if (B < 1 || B > 4096 || n_max < 1 || n_max > 256 || V < 1 || V >= (1 << 30)) return 0;
  return bastion::verify_sample_workspace_bytes(B, n_max, V);
}

int bastion_verify_sample(const void *target_logits, int dtype, int B, int n_max, int V,
                          int64_t ld_row, int b, float temperature, const double *uniforms,
                          const int32_t *n_nodes, const int32_t *parent, const int32_t *token,
                          int32_t *sampled, int32_t *accept_len, int32_t *accept_nodes,
                          int32_t *out_tokens, void *workspace, size_t workspace_bytes,
                          int32_t *status, bastion_stream_t stream) {
  if (!target_logits || !uniforms || !n_nodes || !parent || !token || !sampled || !accept_len ||
      !accept_nodes || !out_tokens || !workspace || !status)
    return BASTION_ERR_NULL;
  if (dtype != BASTION_F32 && dtype != BASTION_BF16) return BASTION_ERR_DTYPE;
  if (B < 1 || B > 4096 || n_max < 1 || n_max > 256 || V < 1 || V >= (1 << 30) || ld_row < V ||
      b < 1 || b > 32 || !(temperature > 0.f) || !(temperature < 1e30f))
    return BASTION_ERR_SIZE;
  const int es = dtype == BASTION_F32 ? 4 : 2;
  if (!aligned(target_logits, es) || !aligned(uniforms, 8) || !aligned(workspace, 256))
    return BASTION_ERR_ALIGN;
  if (workspace_bytes < bastion::verify_sample_workspace_bytes(B, n_max, V)) return BASTION_ERR_WORKSPACE;
  return bastion::launch_verify_sample(target_logits, dtype, B, n_max, V, ld_row, b, temperature,
                                       uniforms, n_nodes, parent, token, sampled, accept_len,
                                       accept_nodes, out_tokens, workspace, status,
                                       (cudaStream_t)stream);
}

int bastion_calibrate_cost(const float *sample_n, const float *sample_ms, int n_samples,
                           double bytes0, double bytes1, double flops0, double flops1, double bw,
                           double peak, double t_draft, int n_max, float *cost_ms, float *params,
                           int32_t *status, bastion_stream_t stream) {
  if (!sample_n || !sample_ms || !cost_ms || !params || !status) return BASTION_ERR_NULL;
  if (n_samples < 1 || n_samples > (1 << 24) || n_max < 1 || n_max > 256) return BASTION_ERR_SIZE;
  const double v[7] = {bytes0, bytes1, flops0, flops1, bw, peak, t_draft};
  for (double x : v)
    if (!(x == x) || x < 0.0 || x > 1e300) return BASTION_ERR_SIZE;
  if (!(bw > 0.0) || !(peak > 0.0)) return BASTION_ERR_SIZE;
  if (!aligned(sample_n, 4) || !aligned(sample_ms, 4) || !aligned(cost_ms, 4) || !aligned(params, 4))
    return BASTION_ERR_ALIGN;
  return bastion::launch_calibrate(sample_n, sample_ms, n_samples, bytes0, bytes1, flops0, flops1,
                                   bw, peak, t_draft, n_max, cost_ms, params, status,
                                   (cudaStream_t)stream);
}

size_t bastion_tree_attention_workspace_bytes(int B, int n_max, int Hq, int Hkv, int D,
                                              int64_t L_cap) {
  if (B < 1 || n_max < 1 || n_max > 256 || Hq < 1 || Hkv < 1 || Hq % Hkv || D != 128 ||
      L_cap < 1)
    return 0;
  return bastion::attention_workspace_bytes(B, n_max, Hq, Hkv, D, L_cap);
}

int bastion_tree_attention(const void *q, const void *k_cache, const void *v_cache, int B,
                           int n_max, int Hq, int Hkv, int D, int64_t L_cap,
                           const int32_t *ctx_len, const int32_t *n_nodes,
                           const uint32_t *anc_mask, float scale, void *out, void *workspace,
                           size_t workspace_bytes, int32_t *status, bastion_stream_t stream) {
  if (!q || !k_cache || !v_cache || !ctx_len || !n_nodes || !anc_mask || !out || !status ||
      !workspace)
    return BASTION_ERR_NULL;
  if (B < 1 || n_max < 1 || n_max > 256 || Hq < 1 || Hkv < 1 || L_cap < 1 || L_cap >= (1LL << 31))
    return BASTION_ERR_SIZE;
  if (Hq % Hkv) return BASTION_ERR_SIZE;
  if (!(scale > 0.f) || !(scale < 1e30f)) return BASTION_ERR_SIZE;  // the kernel takes maxima of raw scores
  if (D != 128 || Hq / Hkv > 8 || 128 % (Hq / Hkv)) return BASTION_ERR_UNSUPPORTED;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
      !aligned(workspace, 256))
    return BASTION_ERR_ALIGN;
  if (workspace_bytes < bastion::attention_workspace_bytes(B, n_max, Hq, Hkv, D, L_cap))
    return BASTION_ERR_WORKSPACE;
  return bastion::launch_attention(q, k_cache, v_cache, B, n_max, Hq, Hkv, D, L_cap, ctx_len,
                                   n_nodes, anc_mask, scale, out, workspace, status,
                                   (cudaStream_t)stream);
}

}  // extern "C"
