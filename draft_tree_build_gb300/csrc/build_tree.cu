// Steps 2-3 of the draft-tree path: best-first prefix-tree expansion under the
// online budget controller, and the emitted tree arrays.
//
// Bastion (gist.science/nl/paper/2605.29727), Methodologie §1 ("Pad-scoren":
// rho(i) = prod_{k<=d(i)} q_k(x_ik)), §2 ("Surrogaat-schatting": A_hat = sum rho;
// "Optimale Constructie": add the valid node with the highest rho), §3
// ("Adaptief Stoppen": grow until S(N) = A_hat(T_N) L_AR / C(N) starts to fall).
//
// One warp builds one request's tree; requests are independent CTAs.
//  * Scores: log rho of a depth-d node = sum over its path of (logit - lse),
//    kept as a 64-bit fixed-point integer with 2^-40 resolution.  A bf16
//    logit (and an fp32 logit of magnitude >= 2^-17) converts exactly, and
//    every path of depth d subtracts the same rounded lse terms, so two paths
//    of equal depth and equal logit sum get identical scores and the tie rule
//    decides between them; across depths the score is within ~2^-36 of the
//    exact value, far inside the 1e-6 band where floating point may decide.
//    A child's score is its parent's plus one table entry
//    lq[d][j] = fix(logit) - fix(lse_{d+1}), so a pop does integer adds only.
//  * Frontier: node p has one pending candidate, its next-ranked child (p, j);
//    with sorted ranks, the best of these is the best candidate overall.  The
//    pending candidate of node p is held in lane p % 32, register slot p / 32,
//    as a 96-bit key: the order-preserving image of the score (two words),
//    then tie bits 0xFFFFFF - (depth<<18 | rank<<8 | parent) so equal scores
//    prefer lower depth, rank and parent; the slot also keeps node p's score.
//    A pop is three redux.sync reductions, two broadcast table loads, two
//    64-bit adds and selects; no lane waits for another.
//  * Stop test before adding candidate c to a tree of N nodes (C > 0):
//    S(N+1) < S(N)  <=>  rho_c C(N) < A_hat (C(N+1) - C(N)), in fp32 with
//    A_hat summed with Kahan compensation; rho_c = exp(hi) (1 + lo) from the
//    float pair nearest the score.
//  * Per-node results and ancestor masks are kept in shared memory during the
//    build and written out, coalesced, after it.
#include "common.cuh"

namespace bastion {

namespace {

constexpr int kBatch = 16;  // global loads in flight per lane while staging

struct TreeArgs {
  const float *topk_logit;
  const int32_t *topk_tok;
  const double *lse;
  int B, b, K, n_max, R, W;
  const int32_t *root_token, *ctx_len;
  const float *cost;
  int cost_per_request;
  const float *l_ar;
  int32_t *n_nodes, *parent, *depth, *pos_id, *token, *rank;
  float *log_rho, *a_hat, *speedup;
  uint32_t *anc_mask;
  int32_t *status;
};

constexpr float kFix = 1099511627776.f;         // 2^40
constexpr float kUnfix = 9.094947017729282e-13f;  // 2^-40
constexpr int64_t kNegFix = -(1ll << 58);         // the score of a -inf logit
constexpr int64_t kInfCut = -(1ll << 57);         // scores below count as -inf
constexpr float kMaxLogit = 131072.f;             // finite logits clamped to 2^17

// Fixed-point images (2^-40 units) of a logit and of an lse value.
__device__ __forceinline__ int64_t fix_logit(float x) {
  if (!(x > -INFINITY)) return kNegFix;  // -inf (and NaN, which K1 flags)
  return __float2ll_rn(fminf(fmaxf(x, -kMaxLogit), kMaxLogit) * kFix);
}
__device__ __forceinline__ int64_t fix_lse(double x) {
  return __double2ll_rn(fmin(fmax(x, -131072.0), 131072.0) * 1099511627776.0);
}

__device__ __forceinline__ uint64_t key_of(int64_t score) {
  return (uint64_t)score ^ 0x8000000000000000ull;
}

// 96-bit key comparison a > b without branches.
__device__ __forceinline__ bool key_gt(uint32_t ah, uint32_t al, uint32_t at, uint32_t bh,
                                       uint32_t bl, uint32_t bt) {
  return (ah > bh) | ((ah == bh) & ((al > bl) | ((al == bl) & (at > bt))));
}

// rho = exp(score) from the float pair nearest the fixed-point score.
__device__ __forceinline__ float rho_of(int64_t score) {
  const float hi = __ll2float_rn(score) * kUnfix;
  const float lo = __ll2float_rn(score - __float2ll_rn(hi * kFix)) * kUnfix;
  const float e = hi < -104.f ? 0.f : expf(hi);
  return fmaf(e, lo, e);
}

// The largest 96-bit key over the warp.
__device__ __forceinline__ void warp_best(uint32_t bh, uint32_t bl, uint32_t bt, uint32_t &mh,
                                          uint32_t &ml, uint32_t &mt) {
  mh = __reduce_max_sync(kFull, bh);
  ml = __reduce_max_sync(kFull, bh == mh ? bl : 0u);
  mt = __reduce_max_sync(kFull, (bh == mh && bl == ml) ? bt : 0u);
}

template <int S>  // register slots per lane: S * 32 >= n_max
__global__ void __launch_bounds__(32) build_tree_kernel(TreeArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  // [n_max] node scores (padded to an even count, so every later array stays
  // 16-byte aligned), then [b * R] the scores' steps
  int64_t *lq = reinterpret_cast<int64_t *>(smem) + ((a.n_max + 1) & ~1);
  int *tk = reinterpret_cast<int *>(lq + a.b * a.R);                 // [b * R] tokens
  float *C = reinterpret_cast<float *>(tk + a.b * a.R);              // [n_max + 1]
  uint32_t *mask = reinterpret_cast<uint32_t *>(C + a.n_max + 1);   // [n_max * W]
  int *nd_par = reinterpret_cast<int *>(mask + a.n_max * a.W);       // [n_max] per node:
  int *nd_dj = nd_par + a.n_max;                                     //   depth << 16 | rank
  float *nd_A = reinterpret_cast<float *>(nd_dj + a.n_max);          //   A_hat after it
  int64_t *nd_sc = reinterpret_cast<int64_t *>(smem);               //   score (first array)

  const int r = blockIdx.x, lane = threadIdx.x;
  const int R = a.R, W = a.W, b = a.b;
  griddep_wait();
  griddep_launch_dependents();
  // ---- stage the request's inputs; every load of a batch is issued before use
  const int ctx = a.ctx_len[r];
  const float L_ar = a.l_ar[r];
  const int root_tok = a.root_token[r];
  const int64_t lse_fix = fix_lse(lane < b ? a.lse[(size_t)r * b + lane] : 0.0);
  const float *cr = a.cost + (a.cost_per_request ? (size_t)r * (a.n_max + 1) : 0);
  float cv[9];  // n_max + 1 <= 257 <= 9 * 32
#pragma unroll
  for (int u = 0; u < 9; ++u) {
    const int i = u * 32 + lane;
    cv[u] = i <= a.n_max ? __ldg(cr + i) : 1.f;
  }
  {
    const int nlg = b * R;
    const float *gl = a.topk_logit + (size_t)r * b * a.K;
    const int32_t *gt = a.topk_tok + (size_t)r * b * a.K;
    const bool vec = R == a.K && (R & 3) == 0 && ((uintptr_t)gl & 15) == 0 &&
                     ((uintptr_t)gt & 15) == 0;
    if (vec) {  // the [b][K] block is contiguous and each 16 bytes lie in one row
      const int n4 = nlg >> 2, r4 = R >> 2;
      for (int base = 0; base < n4; base += 32 * kBatch / 2) {
        float4 v[kBatch / 2];
        int4 t[kBatch / 2];
#pragma unroll
        for (int u = 0; u < kBatch / 2; ++u) {
          const int i = base + u * 32 + lane;
          if (i < n4) {
            v[u] = __ldg(reinterpret_cast<const float4 *>(gl) + i);
            t[u] = __ldg(reinterpret_cast<const int4 *>(gt) + i);
          }
        }
#pragma unroll
        for (int u = 0; u < kBatch / 2; ++u) {
          const int i = base + u * 32 + lane;
          const int64_t ls = __shfl_sync(kFull, lse_fix, min(i, n4 - 1) / r4);
          if (i < n4) {
            const float e[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int64_t f = fix_logit(e[q]);
              lq[4 * i + q] = f == kNegFix ? kNegFix : f - ls;
            }
            reinterpret_cast<int4 *>(tk)[i] = t[u];
          }
        }
      }
    } else {
      for (int base = 0; base < nlg; base += 32 * kBatch) {
        float v[kBatch];
        int t[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          const int idx = base + u * 32 + lane;
          if (idx < nlg) {
            const int d = idx / R, j = idx - d * R;
            v[u] = __ldg(gl + (size_t)d * a.K + j);
            t[u] = __ldg(gt + (size_t)d * a.K + j);
          }
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          const int idx = base + u * 32 + lane;
          const int64_t ls = __shfl_sync(kFull, lse_fix, min(idx, nlg - 1) / R);
          if (idx < nlg) {
            const int64_t f = fix_logit(v[u]);
            lq[idx] = f == kNegFix ? kNegFix : f - ls;
            tk[idx] = t[u];
          }
        }
      }
    }
  }
  bool bad = false;
#pragma unroll
  for (int u = 0; u < 9; ++u) {
    const int i = u * 32 + lane;
    if (i <= a.n_max) {
      C[i] = cv[u];
      if (i >= 1) bad |= !(cv[u] > 0.f) || isinf(cv[u]);
    }
  }
  if (__any_sync(kFull, bad) && lane == 0) atomicOr(&a.status[r], BASTION_STATUS_BAD_COST);
  for (int w = lane; w < W; w += 32) mask[w] = w == 0 ? 1u : 0u;
  __syncwarp();

  // ---- the build; slot s of this lane holds node s * 32 + lane: the key of
  // its pending candidate and the node's own score
  uint32_t kh[S], kl[S], kt[S];
  int64_t sc[S];
#pragma unroll
  for (int s = 0; s < S; ++s) { kh[s] = kl[s] = kt[s] = 0u; sc[s] = 0; }
  if (lane == 0) {  // the root: score 0, pending candidate (0, 0) at depth 1
    const uint64_t k = key_of(lq[0]);
    kh[0] = (uint32_t)(k >> 32);
    kl[0] = (uint32_t)k;
    kt[0] = 0xFFFFFFu - (1u << 18);
  }
  uint32_t bh = kh[0], bl = kl[0], bt = kt[0];
  uint32_t mh, ml, mt;
  warp_best(bh, bl, bt, mh, ml, mt);

  float A_hi = 1.f, A_lo = 0.f;  // A_hat with Kahan compensation
  int N = 1;
  while (N < a.n_max) {
    if ((mh | ml | mt) == 0u) break;  // no candidate left
    const int64_t lr = (int64_t)((((uint64_t)mh << 32) | ml) ^ 0x8000000000000000ull);
    if (lr < kInfCut) break;  // the best candidate has log rho = -inf
    const uint32_t sec = 0xFFFFFFu - mt;
    const int d = (int)(sec >> 18), j = (int)((sec >> 8) & 1023u), p = (int)(sec & 255u);
    const int n = N;
    const int lp = p & 31, sp = p >> 5, ln = n & 31, sn = n >> 5;
    // the winner's rho, the two candidates this pop creates ((p, j + 1) and
    // (n, 0)) and the parent's mask row, all independent of one another
    const float rho = rho_of(lr);
    int64_t sp_score = 0;
#pragma unroll
    for (int s = 0; s < S; ++s) sp_score = s == sp ? sc[s] : sp_score;
    const int jn = j + 1;
    const bool vs = jn < R, vc = d < b;
    const int64_t qs = lq[(d - 1) * R + (vs ? jn : j)];
    const int64_t qc = lq[(vc ? d : d - 1) * R];
    const uint32_t mrow = lane < W ? mask[p * W + lane] : 0u;
    const float Cp = C[N], Cn = C[N + 1];
    const uint64_t ks = key_of(sp_score + qs), kc = key_of(lr + qc);
    const uint32_t ts = 0xFFFFFFu - (((uint32_t)d << 18) | ((uint32_t)jn << 8) | (uint32_t)p);
    const uint32_t tc = 0xFFFFFFu - (((uint32_t)(d + 1) << 18) | (uint32_t)n);
    // the slots change before the stop test: if the build stops they are
    // dropped with it
#pragma unroll
    for (int s = 0; s < S; ++s) {
      const bool up = lane == lp && s == sp;
      const bool un = lane == ln && s == sn;
      kh[s] = up ? (vs ? (uint32_t)(ks >> 32) : 0u) : (un ? (vc ? (uint32_t)(kc >> 32) : 0u) : kh[s]);
      kl[s] = up ? (vs ? (uint32_t)ks : 0u) : (un ? (vc ? (uint32_t)kc : 0u) : kl[s]);
      kt[s] = up ? (vs ? ts : 0u) : (un ? (vc ? tc : 0u) : kt[s]);
      sc[s] = un ? lr : sc[s];
    }
    bh = kh[0]; bl = kl[0]; bt = kt[0];
#pragma unroll
    for (int s = 1; s < S; ++s) {
      const bool g = key_gt(kh[s], kl[s], kt[s], bh, bl, bt);
      bh = g ? kh[s] : bh; bl = g ? kl[s] : bl; bt = g ? kt[s] : bt;
    }
    // the next winner does not depend on the stop test: its reductions
    // overlap the winner's rho (discarded if the build stops here)
    warp_best(bh, bl, bt, mh, ml, mt);
    if (rho * Cp < (A_hi + A_lo) * (Cn - Cp)) break;  // S would decrease: keep T_N

    N = n + 1;
    {
      const float y = rho - A_lo;
      const float t = A_hi + y;
      A_lo = (t - A_hi) - y;
      A_hi = t;
    }
    if (lane == 0) {
      nd_par[n] = p;
      nd_dj[n] = (d << 16) | j;
      nd_sc[n] = lr;
      nd_A[n] = A_hi + A_lo;
    }
    if (lane < W) mask[n * W + lane] = mrow | (lane == (n >> 5) ? (1u << (n & 31)) : 0u);
  }
  __syncwarp();

  // ---- outputs, coalesced
  const size_t nb = (size_t)r * a.n_max;
  if (lane == 0) a.n_nodes[r] = N;
  for (int i = lane; i < N; i += 32) {
    const size_t o = nb + i;
    if (i == 0) {
      a.parent[o] = -1;
      a.depth[o] = 0;
      a.pos_id[o] = ctx;
      a.token[o] = root_tok;
      a.rank[o] = -1;
      a.log_rho[o] = 0.f;
      a.a_hat[o] = 1.f;
      a.speedup[o] = L_ar / C[1];
    } else {
      const int dj = nd_dj[i], d = dj >> 16, j = dj & 0xffff;
      const float Ah = nd_A[i];
      a.parent[o] = nd_par[i];
      a.depth[o] = d;
      a.pos_id[o] = ctx + d;
      a.token[o] = tk[(d - 1) * R + j];
      a.rank[o] = j;
      a.log_rho[o] = __ll2float_rn(nd_sc[i]) * kUnfix;
      a.a_hat[o] = Ah;
      a.speedup[o] = Ah * L_ar / C[i + 1];
    }
  }
  for (int q = lane; q < N * W; q += 32) a.anc_mask[nb * W + q] = mask[q];
}

template <int S>
void launch_s(const TreeArgs &a, size_t smem, cudaStream_t stream) {
  if (smem > 48 * 1024)
    cudaFuncSetAttribute(build_tree_kernel<S>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  launch_pdl(build_tree_kernel<S>, dim3(a.B), dim3(32), smem, stream, a);
}

}  // namespace

int launch_build_tree(const float *topk_logit, const int32_t *topk_tok, const double *lse, int B,
                      int b, int K, int n_max, const int32_t *root_token, const int32_t *ctx_len,
                      const float *cost_ms, int cost_per_request, const float *l_ar,
                      int32_t *n_nodes, int32_t *parent, int32_t *depth, int32_t *pos_id,
                      int32_t *token, int32_t *rank, float *log_rho, float *a_hat, float *speedup,
                      uint32_t *anc_mask, int32_t *status, cudaStream_t stream) {
  TreeArgs a;
  a.topk_logit = topk_logit;
  a.topk_tok = topk_tok;
  a.lse = lse;
  a.B = B;
  a.b = b;
  a.K = K;
  a.n_max = n_max;
  a.R = K < n_max ? K : n_max;
  a.W = (n_max + 31) / 32;
  a.root_token = root_token;
  a.ctx_len = ctx_len;
  a.cost = cost_ms;
  a.cost_per_request = cost_per_request;
  a.l_ar = l_ar;
  a.n_nodes = n_nodes;
  a.parent = parent;
  a.depth = depth;
  a.pos_id = pos_id;
  a.token = token;
  a.rank = rank;
  a.log_rho = log_rho;
  a.a_hat = a_hat;
  a.speedup = speedup;
  a.anc_mask = anc_mask;
  a.status = status;
  const size_t smem = (size_t)((n_max + 1) & ~1) * 8 + (size_t)b * a.R * 12 + (size_t)(n_max + 1) * 4 +
                      (size_t)n_max * a.W * 4 + (size_t)n_max * 12;
  if (n_max <= 32) launch_s<1>(a, smem, stream);
  else if (n_max <= 64) launch_s<2>(a, smem, stream);
  else if (n_max <= 128) launch_s<4>(a, smem, stream);
  else launch_s<8>(a, smem, stream);
  return cudaGetLastError() == cudaSuccess ? BASTION_OK : BASTION_ERR_LAUNCH;
}

}  // namespace bastion
