// Steps 2-3 of the draft-tree path: best-first prefix-tree expansion under the
// online budget controller, and the emitted tree arrays.
//
// Bastion (gist.science/nl/paper/2605.29727), Methodologie §1 ("Pad-scoren":
// rho(i) = prod_{k<=d(i)} q_k(x_ik)), §2 ("Surrogaat-schatting": A_hat = sum rho;
// "Optimale Constructie": add the valid node with the highest rho), §3
// ("Adaptief Stoppen": grow until S(N) = A_hat(T_N) L_AR / C(N) starts to fall).
//
// One warp builds one request's tree; requests are independent CTAs.
//  * Frontier: each tree node p has at most one pending candidate, its next
//    ranked child (p, j).  Because the children's q are sorted, the best
//    candidate of the full frontier is always among these.  The pending
//    candidate of node p lives in register slot p/32 of lane p%32 as a 96-bit
//    key: order-preserving image of log rho (fp64), then the tie bits
//    0xFFFFFF - (depth<<18 | rank<<8 | parent), so that equal scores prefer the
//    lower depth, rank and parent.  Each lane caches its best slot; a pop is
//    three redux.sync max reductions over the warp.
//  * log rho of a depth-d candidate = (fp64 sum of its path's logits, root
//    down) - Lam[d], Lam[d] = lse_1 + ... + lse_d (fp64, in that order).
//  * Stop test before adding the best candidate c to a tree of N nodes:
//    S(N+1) < S(N)  <=>  rho_c C(N) < A_hat (C(N+1) - C(N))   (C > 0).
//  * Ancestor masks are built in shared memory and stored row by row.
#include "common.cuh"

namespace bastion {

namespace {

constexpr int kSlots = 8;  // 8 slots x 32 lanes = 256 nodes

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

__device__ __forceinline__ bool key_gt(uint32_t ah, uint32_t al, uint32_t at, uint32_t bh,
                                       uint32_t bl, uint32_t bt) {
  if (ah != bh) return ah > bh;
  if (al != bl) return al > bl;
  return at > bt;
}

__device__ __forceinline__ void cand_key(double lr, int d, int j, int p, uint32_t &h, uint32_t &l,
                                         uint32_t &t) {
  const uint64_t o = ord_f64(lr);
  h = (uint32_t)(o >> 32);
  l = (uint32_t)o;
  t = 0xFFFFFFu - (((uint32_t)d << 18) | ((uint32_t)j << 8) | (uint32_t)p);
}

// rho = exp(log rho) from an fp32 exp of the leading part times (1 + the
// remainder): relative error a few fp32 ulps; 0 far below fp32 range.
__device__ __forceinline__ double rho_of(double lr) {
  if (lr < -150.0) return 0.0;
  const float hi = (float)lr;
  const float lo = (float)(lr - (double)hi);
  return (double)expf(hi) * (1.0 + (double)lo);
}

__global__ void __launch_bounds__(32) build_tree_kernel(TreeArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  double *Lsum = reinterpret_cast<double *>(smem);         // [n_max] path logit sums
  double *Lam = Lsum + a.n_max;                             // [33]
  float *C = reinterpret_cast<float *>(Lam + 33);           // [n_max + 1]
  uint32_t *mask = reinterpret_cast<uint32_t *>(C + a.n_max + 1);  // [n_max * W]
  float *lg = reinterpret_cast<float *>(mask + a.n_max * a.W);     // [b * R]

  const int r = blockIdx.x, lane = threadIdx.x;
  const int R = a.R, W = a.W;
  for (int idx = lane; idx < a.b * R; idx += 32) {
    const int d = idx / R, j = idx - d * R;
    lg[idx] = a.topk_logit[((size_t)r * a.b + d) * a.K + j];
  }
  const float *cr = a.cost + (a.cost_per_request ? (size_t)r * (a.n_max + 1) : 0);
  bool bad = false;
  for (int i = lane; i <= a.n_max; i += 32) {
    const float c = cr[i];
    C[i] = c;
    if (i >= 1) bad |= !(c > 0.f) || isinf(c);
  }
  if (__any_sync(kFull, bad) && lane == 0) atomicOr(&a.status[r], BASTION_STATUS_BAD_COST);
  if (lane == 0) {
    double acc = 0.0;
    Lam[0] = 0.0;
    for (int d = 1; d <= a.b; ++d) {
      acc = acc + a.lse[(size_t)r * a.b + d - 1];
      Lam[d] = acc;
    }
  }
  const int ctx = a.ctx_len[r];
  const double L = (double)a.l_ar[r];
  const size_t nb = (size_t)r * a.n_max;
  if (lane == 0) {
    a.parent[nb] = -1;
    a.depth[nb] = 0;
    a.pos_id[nb] = ctx;
    a.token[nb] = a.root_token[r];
    a.rank[nb] = -1;
    a.log_rho[nb] = 0.f;
    a.a_hat[nb] = 1.f;
    a.speedup[nb] = a.n_max >= 1 ? (float)(L / (double)C[1]) : 0.f;
    Lsum[0] = 0.0;
  }
  for (int w = lane; w < W; w += 32) {
    const uint32_t m = w == 0 ? 1u : 0u;
    mask[w] = m;
    a.anc_mask[nb * W + w] = m;
  }
  __syncwarp();

  uint32_t kh[kSlots], kl[kSlots], kt[kSlots];
#pragma unroll
  for (int s = 0; s < kSlots; ++s) kh[s] = kl[s] = kt[s] = 0u;
  uint32_t bh = 0u, bl = 0u, bt = 0u;
  if (lane == 0) {
    cand_key((double)lg[0] - Lam[1], 1, 0, 0, kh[0], kl[0], kt[0]);
    bh = kh[0]; bl = kl[0]; bt = kt[0];
  }

  double A = 1.0;
  int N = 1;
  while (N < a.n_max) {
    const uint32_t mh = __reduce_max_sync(kFull, bh);
    const uint32_t ml = __reduce_max_sync(kFull, bh == mh ? bl : 0u);
    const uint32_t mt = __reduce_max_sync(kFull, (bh == mh && bl == ml) ? bt : 0u);
    if ((mh | ml | mt) == 0u) break;  // no candidate left
    const double lr = unord_f64(((uint64_t)mh << 32) | ml);
    if (lr == -INFINITY) break;
    const uint32_t sec = 0xFFFFFFu - mt;
    const int d = (int)(sec >> 18), j = (int)((sec >> 8) & 1023u), p = (int)(sec & 255u);
    const double rho = rho_of(lr);
    const double Cp = (double)C[N], Cn = (double)C[N + 1];
    if (rho * Cp < A * (Cn - Cp)) break;  // S would decrease: keep T_N

    const int n = N;
    const double ls = Lsum[p] + (double)lg[(d - 1) * R + j];
    A += rho;
    N = n + 1;
    if (lane == 0) {
      Lsum[n] = ls;
      const size_t o = nb + n;
      a.parent[o] = p;
      a.depth[o] = d;
      a.pos_id[o] = ctx + d;
      a.token[o] = a.topk_tok[((size_t)r * a.b + d - 1) * a.K + j];
      a.rank[o] = j;
      a.log_rho[o] = (float)lr;
      a.a_hat[o] = (float)A;
      a.speedup[o] = (float)(A * L / Cn);
    }
    for (int w = lane; w < W; w += 32) {
      const uint32_t m = mask[p * W + w] | (w == (n >> 5) ? (1u << (n & 31)) : 0u);
      mask[n * W + w] = m;
      a.anc_mask[(nb + n) * W + w] = m;
    }
    bool touched = false;
    if (lane == (p & 31)) {  // node p's next-ranked child replaces (p, j)
      uint32_t h2 = 0u, l2 = 0u, t2 = 0u;
      if (j + 1 < R) cand_key(Lsum[p] + (double)lg[(d - 1) * R + j + 1] - Lam[d], d, j + 1, p, h2, l2, t2);
      const int s0 = p >> 5;
#pragma unroll
      for (int s = 0; s < kSlots; ++s)
        if (s == s0) { kh[s] = h2; kl[s] = l2; kt[s] = t2; }
      touched = true;
    }
    if (d < a.b && lane == (n & 31)) {  // the new node's first child
      uint32_t h3, l3, t3;
      cand_key(ls + (double)lg[d * R] - Lam[d + 1], d + 1, 0, n, h3, l3, t3);
      const int s1 = n >> 5;
#pragma unroll
      for (int s = 0; s < kSlots; ++s)
        if (s == s1) { kh[s] = h3; kl[s] = l3; kt[s] = t3; }
      touched = true;
    }
    if (touched) {
      bh = kh[0]; bl = kl[0]; bt = kt[0];
#pragma unroll
      for (int s = 1; s < kSlots; ++s)
        if (key_gt(kh[s], kl[s], kt[s], bh, bl, bt)) { bh = kh[s]; bl = kl[s]; bt = kt[s]; }
    }
    __syncwarp();
  }
  if (lane == 0) a.n_nodes[r] = N;
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
  const size_t smem = (size_t)n_max * 8 + 33 * 8 + (size_t)(n_max + 1) * 4 +
                      (size_t)n_max * a.W * 4 + (size_t)b * a.R * 4;
  if (smem > 48 * 1024)
    cudaFuncSetAttribute(build_tree_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  build_tree_kernel<<<B, 32, smem, stream>>>(a);
  return cudaGetLastError() == cudaSuccess ? BASTION_OK : BASTION_ERR_LAUNCH;
}

}  // namespace bastion
