/*
 * bastion.h -- C ABI of the GB300 (sm_103a) draft-tree hot path.
 *
 * The method: "Bastion: Budget-Aware Speculative Decoding with Tree-structured
 * Block Diffusion Drafting" (gist.science/nl/paper/2605.29727, technical
 * summary, "Methodologie" §1-§3; same text on gist.science/fr/paper/2605.29727).
 * A block-diffusion drafter emits one marginal q_k per block position in one
 * forward pass; a prefix tree of candidate continuations is grown best-first by
 * path score rho(i) = prod_{k<=d(i)} q_k(x_ik) until the estimated speedup
 * S(N) = A_hat(T_N) * L_AR / C(N), A_hat = sum rho, starts to fall; the target
 * verifies the tree in one parallel pass (tree-masked attention) and greedy
 * (temperature 0) acceptance keeps the longest matching root path plus one
 * bonus token.
 *
 * Conventions shared by every entry point:
 *  - All tensors are caller-owned DEVICE pointers, row-major, with the shapes
 *    given at each function.  The library allocates nothing and keeps no
 *    global mutable state; every call is asynchronous on the caller's stream.
 *  - Return value: BASTION_OK, or a negative BASTION_ERR_* code when an
 *    argument check on the host fails (nothing is launched then), or
 *    BASTION_ERR_LAUNCH when the launch itself reports an error.
 *  - Data-dependent problems found on the device (a NaN or +inf logit, a
 *    non-positive cost, a tree too large for the KV cache, a bounded wait that
 *    ran out) are OR-ed as BASTION_STATUS_* bits into status[r] of the
 *    request concerned; the caller zeroes status before the calls it wants to
 *    check.  The outputs of a request with a status bit set are unspecified.
 *    No kernel traps or asserts.
 *  - Workspace: functions that take one need at least *_workspace_bytes()
 *    bytes, 256-byte aligned, ZERO-FILLED before its first use.  It holds
 *    per-call partial results and arrival counters; every call that completes
 *    returns the counters to zero, so the same workspace serves the next call
 *    without clearing.  Calls that may run concurrently need separate
 *    workspaces.
 *  - dtype: BASTION_F32 (float) or BASTION_BF16 (bfloat16 bits).
 */
#ifndef BASTION_H_
#define BASTION_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *bastion_stream_t; /* the same handle as cudaStream_t */

enum { BASTION_F32 = 0, BASTION_BF16 = 1 };

enum {
  BASTION_OK = 0,
  BASTION_ERR_NULL = -1,        /* a required pointer is null */
  BASTION_ERR_SIZE = -2,        /* a size, count or stride is out of range */
  BASTION_ERR_DTYPE = -3,       /* unknown dtype */
  BASTION_ERR_ALIGN = -4,       /* a pointer misses its documented alignment */
  BASTION_ERR_WORKSPACE = -5,   /* workspace missing or too small */
  BASTION_ERR_UNSUPPORTED = -6, /* valid but not implemented (e.g. head dim) */
  BASTION_ERR_LAUNCH = -7       /* the CUDA launch reported an error */
};

enum {
  BASTION_STATUS_NONFINITE = 1,    /* a NaN or +inf logit in the request's rows */
  BASTION_STATUS_EMPTY_ROW = 2,    /* a drafter row with no finite logit */
  BASTION_STATUS_BAD_COST = 4,     /* some C(N) <= 0 or not finite */
  BASTION_STATUS_KV_OVERFLOW = 8,  /* ctx_len + n_nodes > L_cap, or ctx_len < 0 */
  BASTION_STATUS_BAD_TREE = 16,    /* n_nodes outside [1, n_max] */
  BASTION_STATUS_BAD_WEIGHT = 32,  /* a mixture weight pi is negative or not finite */
  BASTION_STATUS_TIMEOUT = 1 << 30 /* a bounded device wait ran out */
};

/* Library version string ("bastion-gb300 x.y.z sm_103a"). */
const char *bastion_version(void);

/* Text for a BASTION_ERR_* return code or a single BASTION_STATUS_* bit. */
const char *bastion_status_string(int code);

/* ---------------------------------------------------------------------------
 * Step 1 -- softmax + top-K marginals.
 * Methodologie §1 ("positie-afhankelijke marginaalverdelingen {q_k}"): for
 * every drafter row (request r, block position k) it forms q_k = softmax(l_k)
 * and ranks the vocabulary by q_k (equivalently by logit), ties broken by the
 * lower token id; the K best are kept.
 *
 * logits     [B, b, V] at row stride ld_row elements (ld_row >= V), dtype as
 *            given.  Any address is accepted; 16-byte aligned rows read fastest.
 * topk_logq  [B, b, K] float  log q_k of each kept token, l - lse rounded once.
 *            May be NULL.
 * topk_logit [B, b, K] float  the kept logits exactly as given (fp32 value).
 * topk_tok   [B, b, K] int32  token ids, rank order.
 * lse        [B, b] double    log sum_v exp(l_v), within ~2e-6 absolute
 *                             (fp32 exponentials, compensated sums, fp64 log).
 * status     [B] int32        OR-ed BASTION_STATUS_* bits.
 * Limits: B >= 1, 1 <= b <= 32, 1 <= K <= min(V, 1024), V < 2^30.
 * Workspace: bastion_topk_marginals_workspace_bytes(B, b, V, K) bytes.
 * One kernel launch.  From two rows per SM on, one CTA streams each row; with
 * fewer rows a cluster of CTAs shares each row.  Tokens and logits do not
 * depend on which kernel ran, lse only within its stated bound;
 * BASTION_TOPK_PATH=stream|cluster in the environment forces one of them where
 * it applies (for tests).
 */
size_t bastion_topk_marginals_workspace_bytes(int B, int b, int V, int K);
int bastion_topk_marginals(const void *logits, int dtype, int B, int b, int V, int64_t ld_row,
                           int K, float *topk_logq, float *topk_logit, int32_t *topk_tok,
                           double *lse, void *workspace, size_t workspace_bytes,
                           int32_t *status, bastion_stream_t stream);

/* ---------------------------------------------------------------------------
 * Step 1 fused with the drafter's output layer: the top-K marginals of the
 * logits l_k = W h_k, formed on the tensor cores and never written out.
 * Methodologie §1: one forward pass of the block-diffusion drafter yields the
 * position-wise marginals q_k = softmax(l_k); W is its output embedding and
 * h_k the final hidden state of block position k.
 *
 * hidden     [B, b, H] bf16, row-major, 16-byte aligned; H a multiple of 64
 *            (BASTION_ERR_UNSUPPORTED otherwise).
 * weight     [V, H] bf16, row-major, 16-byte aligned.
 * Outputs:   as bastion_topk_marginals, for the logits as accumulated (fp32,
 *            bf16 products summed on the tensor cores): topk_logq (may be
 *            NULL), topk_logit, topk_tok [B, b, K] in rank order (logit desc,
 *            token asc), lse [B, b] double, status [B].  Each logit differs
 *            from the exact dot product by the accumulation's rounding, well
 *            inside 2^-16 sum_i |W[v,i] h[i]|, so tokens whose exact logits lie
 *            closer than that may come in either order.
 * Limits: B, b >= 1, B*b <= 2^24, 1 <= K <= min(V, 64), V < 2^31, H <= 2^20.
 * Workspace: bastion_lm_head_topk_workspace_bytes(B, b, V, K) bytes, 256-byte
 * aligned, zero-filled before its first use; every call leaves it so.  Calls
 * that share a workspace must not overlap on the GPU.  Two launches (the GEMM
 * with its per-share top-K, then the per-row merge).
 */
size_t bastion_lm_head_topk_workspace_bytes(int B, int b, int V, int K);
int bastion_lm_head_topk(const void *hidden, const void *weight, int B, int b, int H, int V, int K,
                         float *topk_logq, float *topk_logit, int32_t *topk_tok, double *lse,
                         void *workspace, size_t workspace_bytes, int32_t *status,
                         bastion_stream_t stream);

/* ---------------------------------------------------------------------------
 * Steps 2-3 -- best-first tree expansion under the online budget controller,
 * and the tree arrays.
 * Methodologie §1 ("Pad-scoren": rho = prod q_k), §2 ("Surrogaat-schatting":
 * A_hat = sum rho; "Optimale Constructie": always add the valid node with the
 * highest rho), §3 ("Adaptief Stoppen": grow until S(N) = A_hat*L_AR/C(N)
 * starts to decrease).
 *
 * Node 0 is the root (the last committed token, root_token[r]) at depth 0 with
 * rho = 1, counted in N and A_hat.  The children of a depth-d node are the K
 * ranked tokens of q_{d+1}; a node's next candidate child is its next-ranked
 * token.  Candidates are ordered by log rho (descending), then depth, rank and
 * parent index (ascending).  log rho of a depth-d node is the sum over its
 * path of (logit - lse_k), formed in 64-bit fixed point with 2^-40 resolution:
 * exact for bf16 logits (and fp32 logits of magnitude >= 2^-17), so paths of
 * equal depth and equal logit sum tie exactly and the tie rule decides; finite
 * logits are clamped to +-2^17.  From N = 1 (root only),
 * the best candidate is added as node N while S(N+1) >= S(N); the build stops
 * at the first strict decrease, when no candidate is left, or at n_max nodes.
 * One warp builds one request's tree.
 *
 * topk_logit, topk_tok [B, b, K], lse [B, b]: the outputs of step 1.
 * root_token, ctx_len [B] int32.
 * cost_ms    [Bc, n_max+1] float: entry N is C(N) = T_draft + T_verify(N) in
 *            ms for a tree of N nodes; Bc = B when cost_per_request != 0, else 1.
 * l_ar       [B] float: L_AR in ms (it scales S and does not move the stop).
 * Outputs:   n_nodes [B]; per node [B, n_max] (rows >= n_nodes untouched):
 *            parent (root -1), depth, pos_id (= ctx_len + depth), token, rank
 *            (root -1), log_rho (float), a_hat (A_hat of nodes 0..n), speedup
 *            (S at size n+1); anc_mask [B, n_max, W] uint32 with
 *            W = ceil(n_max/32): bit t%32 of word t/32 of node i is set iff node
 *            t is node i or one of its ancestors.  Node order is pop order
 *            (parent[i] < i).
 * Limits: B >= 1, 1 <= b <= 32, 1 <= K <= 1024, 1 <= n_max <= 256.
 */
int bastion_build_tree(const float *topk_logit, const int32_t *topk_tok, const double *lse,
                       int B, int b, int K, int n_max, const int32_t *root_token,
                       const int32_t *ctx_len, const float *cost_ms, int cost_per_request,
                       const float *l_ar, int32_t *n_nodes, int32_t *parent, int32_t *depth,
                       int32_t *pos_id, int32_t *token, int32_t *rank, float *log_rho,
                       float *a_hat, float *speedup, uint32_t *anc_mask, int32_t *status,
                       bastion_stream_t stream);

/* ---------------------------------------------------------------------------
 * Best-first draft tree on a latent-mixture proposal (DBlast, "Methodologie" 1:
 * q_dep(x_1..b | y) = sum_z q(z|y) prod_i q_i(x_i | y, z), grown with Bastion's
 * §1-§3 controller).  The prefix score is the mixture probability
 * rho(x_1..d) = sum_z pi_z prod_{k<=d} q_k^z(x_k); a token outside branch z's
 * list at position k has q_k^z = 0; the children of a depth-d node are the
 * union over z of the branches' tokens at position d+1.  Candidates are
 * ordered by log rho (descending), then depth and token id (ascending).  The
 * stop rule is bastion_build_tree's.  Per-branch path scores are 64-bit fixed
 * point; the mixture sum over the branches is formed in fp32 with log rho
 * within about (5 + Z/2) 2^-23 of exact, so where two candidates lie within
 * 1e-5 of each other in log rho, or a stop test within 1e-5 (relative) of its
 * boundary, either choice is a correct result.
 *
 * topk_logit, topk_tok [B, Z, b, K], lse [B, Z, b] (8-byte aligned): step 1
 *            run per branch; each branch lists a token at most once per
 *            position (otherwise the results are undefined); no token equals
 *            INT32_MIN.  pi [B, Z] double (8-byte aligned), each row the
 *            branch weights q(z|y), summing to 1.  A weight that is negative,
 *            NaN or infinite sets BASTION_STATUS_BAD_WEIGHT in status[r] and
 *            counts as 0 in that request's tree.
 * root_token, ctx_len, cost_ms, cost_per_request, l_ar: as bastion_build_tree.
 * Outputs:   as bastion_build_tree without rank: n_nodes [B]; parent, depth,
 *            pos_id, token, log_rho, a_hat, speedup [B, n_max];
 *            anc_mask [B, n_max, ceil(n_max/32)].
 * Workspace: bastion_build_tree_mixture_workspace_bytes(B, Z, b, K, n_max)
 *            bytes, 256-byte aligned: each request's tables, written by a
 *            staging launch and read by the build launch (two launches on the
 *            stream; calls sharing a workspace must not overlap on the GPU).
 * Limits: 1 <= Z <= 32, 1 <= K <= 1024, 1 <= b <= 32, 1 <= n_max <= 256
 * (BASTION_ERR_SIZE otherwise); one request's tables, about
 * 18 b Z K + 16 n_max (Z + 2 + Z K / 32) bytes (with Z <= 8 and room, a
 * faster layout of about b Z K (18 + 6 Zp) bytes, Zp = Z rounded up to 1, 2,
 * 4 or 8), must fit in 227 KB of shared memory (BASTION_ERR_UNSUPPORTED
 * otherwise): b = 16 allows Z K up to about 600 at n_max = 128, e.g. Z = 4
 * with K = 128, or Z = 8 with K = 64.
 */
size_t bastion_build_tree_mixture_workspace_bytes(int B, int Z, int b, int K, int n_max);

int bastion_build_tree_mixture(const float *topk_logit, const int32_t *topk_tok, const double *lse,
                               const double *pi, int B, int Z, int b, int K, int n_max,
                               const int32_t *root_token, const int32_t *ctx_len,
                               const float *cost_ms, int cost_per_request, const float *l_ar,
                               int32_t *n_nodes, int32_t *parent, int32_t *depth, int32_t *pos_id,
                               int32_t *token, float *log_rho, float *a_hat, float *speedup,
                               uint32_t *anc_mask, void *workspace, size_t workspace_bytes,
                               int32_t *status, bastion_stream_t stream);

/* ---------------------------------------------------------------------------
 * Tree-masked GQA attention of the tree's query tokens against the KV cache
 * (the target's parallel verification pass over the whole tree,
 * "Probleemstelling" and Methodologie §2).
 *
 * O[r,i,h] = sum_j softmax_j(scale * Q[r,i,h] . K[r,j,h/G]) V[r,j,h/G],
 * G = Hq/Hkv.  Key slot j < ctx_len[r] is visible to every query; tree slot
 * ctx_len[r] + t (t < n_nodes[r]) is visible to query i iff bit t of
 * anc_mask[r,i]; other slots are not visible.  Rows i >= n_nodes[r] of out
 * are left untouched.  bf16 inputs, fp32 accumulation, bf16 output (RNE).
 *
 * q        [B, n_max, Hq, D] bf16; k_cache, v_cache [B, L_cap, Hkv, D] bf16,
 *          with the tree's keys/values at slots ctx_len .. ctx_len+n_nodes-1;
 *          all 16-byte aligned.
 * out      [B, n_max, Hq, D] bf16.
 * scale    the softmax scale (1/sqrt(D) for standard attention): finite and
 *          > 0, else BASTION_ERR_SIZE.
 * Limits: D = 128, Hq % Hkv == 0, Hq/Hkv in {1, 2, 4, 8}, 1 <= n_max <= 256.
 * Workspace: bastion_tree_attention_workspace_bytes(...) bytes.
 */
size_t bastion_tree_attention_workspace_bytes(int B, int n_max, int Hq, int Hkv, int D,
                                              int64_t L_cap);
int bastion_tree_attention(const void *q, const void *k_cache, const void *v_cache, int B,
                           int n_max, int Hq, int Hkv, int D, int64_t L_cap,
                           const int32_t *ctx_len, const int32_t *n_nodes,
                           const uint32_t *anc_mask, float scale, void *out, void *workspace,
                           size_t workspace_bytes, int32_t *status, bastion_stream_t stream);

/* ---------------------------------------------------------------------------
 * The cost model of step 2, calibrated on the device.  "Methodologie" §3,
 * "Latentiemodellering": T_verify(N) comes from a hardware-aware roofline model
 * of memory bandwidth and compute, calibrated with observed runtimes.  Here
 *   roof(N)   = max((bytes0 + bytes1 N) / bw, (flops0 + flops1 N) / peak)
 * (units chosen so that roof is in ms, e.g. bytes per ms and flop per ms), and
 * the calibration is the least-squares line T_verify = alpha roof(N) + beta
 * through the observed samples (sample_n[k] tree nodes, sample_ms[k] ms); with
 * no spread in the samples' roofline values alpha = 1 and beta is the mean
 * residual.  Output: cost_ms [n_max + 1] float, C(N) = t_draft + alpha roof(N)
 * + beta, the single-row table bastion_build_tree reads (cost_per_request = 0);
 * params [2] float = {alpha, beta}.  Sums in fp64, one CTA.
 * status [1] int32: BASTION_STATUS_BAD_COST if a sample is non-finite or a
 * C(N), N >= 1, is not positive and finite.
 * Limits: 1 <= n_samples <= 2^24, 1 <= n_max <= 256; the six roofline
 * constants and t_draft finite and >= 0, bw and peak > 0.  One kernel launch.
 */
int bastion_calibrate_cost(const float *sample_n, const float *sample_ms, int n_samples,
                           double bytes0, double bytes1, double flops0, double flops1, double bw,
                           double peak, double t_draft, int n_max, float *cost_ms, float *params,
                           int32_t *status, bastion_stream_t stream);

/* ---------------------------------------------------------------------------
 * Step 4 -- greedy (temperature 0) verification ("Experimentele Resultaten":
 * greedy decoding).  For every tree node i < n_nodes[r] the target's greedy
 * token is argmax_v target[r,i,v] (ties: lowest v).  From the root, the child
 * whose token equals the current node's greedy token is accepted and becomes
 * the current node; the walk ends at the first node without such a child, and
 * that node's greedy token is the bonus token.
 *
 * target_logits [B, n_max, V] at row stride ld_row elements, dtype as given:
 *            device memory, or pinned (page-locked) host memory, which the
 *            sweep reads in place over the host link: only the rows of the
 *            tree's nodes cross it, and no host-side copy or synchronisation
 *            is needed between building the tree and verifying it.
 * n_nodes [B], parent/token [B, n_max]: the tree of step 3.
 * Outputs: argmax [B, n_max] (rows >= n_nodes untouched); accept_len [B]
 *          (0..b); accept_nodes [B, b+1] (root 0, then the accepted nodes,
 *          then -1); out_tokens [B, b+1] (accepted tokens, the bonus, then -1).
 * Limits: 1 <= B <= 4096, 1 <= n_max <= 256, 1 <= b <= 32, V < 2^30.
 * Workspace: bastion_verify_greedy_workspace_bytes(B, n_max, V) bytes.
 */
size_t bastion_verify_greedy_workspace_bytes(int B, int n_max, int V);
int bastion_verify_greedy(const void *target_logits, int dtype, int B, int n_max, int V,
                          int64_t ld_row, int b, const int32_t *n_nodes, const int32_t *parent,
                          const int32_t *token, int32_t *argmax, int32_t *accept_len,
                          int32_t *accept_nodes, int32_t *out_tokens, void *workspace,
                          size_t workspace_bytes, int32_t *status, bastion_stream_t stream);

/* ---------------------------------------------------------------------------
 * Step 4 at temperature T > 0 -- stochastic verification.  The pages evaluate
 * greedy decoding only ("Experimentele Resultaten"; DBlast, introduction:
 * sampled decoding is the regime that matters).  For a tree of deterministic
 * candidates the lossless reading is taken: the target's token at node i is a
 * draw from softmax(target[r,i,:] / T) by inverse transform with the caller's
 * uniform u = uniforms[r,i] in [0, 1) -- the smallest v whose cumulative
 * weight sum_{w <= v} exp(l_w / T) exceeds u times the row's total -- and the
 * greedy walk runs over the draws (the bonus is the draw at the last accepted
 * node).  Every emitted token is then a draw from the target's conditional.
 *
 * The cumulative weights are formed in fp32 (compensated across 4 KB items)
 * with fp32 exponentials: a draw within ~1e-6 of the row's total from a
 * neighbouring token's interval may land on that neighbour.
 * uniforms [B, n_max] double (8-byte aligned), caller-generated.
 * Other arguments, outputs and limits as bastion_verify_greedy; sampled
 * [B, n_max] holds the draws (rows >= n_nodes untouched).  temperature in
 * (0, 1e30).  NaN / +inf logits set BASTION_STATUS_NONFINITE, a row without a
 * finite logit BASTION_STATUS_EMPTY_ROW (its draw is token 0).
 * Workspace: bastion_verify_sample_workspace_bytes(B, n_max, V) bytes.
 * Three kernel launches (a sweep of the live rows, the draws, the walk).
 */
size_t bastion_verify_sample_workspace_bytes(int B, int n_max, int V);
int bastion_verify_sample(const void *target_logits, int dtype, int B, int n_max, int V,
                          int64_t ld_row, int b, float temperature, const double *uniforms,
                          const int32_t *n_nodes, const int32_t *parent, const int32_t *token,
                          int32_t *sampled, int32_t *accept_len, int32_t *accept_nodes,
                          int32_t *out_tokens, void *workspace, size_t workspace_bytes,
                          int32_t *status, bastion_stream_t stream);

/* ---------------------------------------------------------------------------
 * Greedy verification without a workspace, for callers that cannot allocate.
 * The pages have no counterpart: this is a deployment variant of the call
 * above, not a step of the method.
 *
 * Some callers cannot call cudaMalloc or have memory allocated for them (a
 * serving loop that must not touch the allocator after start-up, code inside a
 * framework that owns the allocator, a plug-in that only receives input and
 * output pointers).  This entry point takes the same arguments and gives the
 * same results as bastion_verify_greedy, but its scratch is a fixed 128 KiB
 * array compiled into the library, which every GPU that loads the library
 * holds until the process exits; it calls no cudaMalloc or cudaFree.
 * Limits: B <= 4096 and B * n_max <= 16384 (e.g. 64 requests x 256 nodes);
 * larger sizes return BASTION_ERR_SIZE without launching.
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current); make that first call
 * before any stream capture.  Each call clears the part of the array it uses
 * (cudaMemsetAsync on the caller's stream) and then launches the verify kernel.
 * All calls share the one array: calls that can overlap on the GPU (other
 * streams, other host threads) race on it and must be serialised by the caller.
 */
int bastion_verify_greedy_noalloc(const void *target_logits, int dtype, int B, int n_max, int V,
                                  int64_t ld_row, int b, const int32_t *n_nodes,
                                  const int32_t *parent, const int32_t *token, int32_t *argmax,
                                  int32_t *accept_len, int32_t *accept_nodes, int32_t *out_tokens,
                                  int32_t *status, bastion_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* BASTION_H_ */
