// Steps 2-3 of the draft-tree path: best-first prefix-tree expansion under the
// online budget controller, and the emitted tree arrays.
//
// Bastion (gist.science/nl/paper/2605.29727), Methodologie §1 ("Pad-scoren":
// rho(i) = prod_{k<=d(i)} q_k(x_ik)), §2 ("Surrogaat-schatting": A_hat = sum rho;
// "Optimale Constructie": add the valid node with the highest rho), §3
// ("Adaptief Stoppen": grow until S(N) = A_hat(T_N) L_AR / C(N) starts to fall).
//
// One warp builds one request's tree; requests are independent CTAs.
//  * Scores: log rho of a depth-d node = L - Lam[d], L = the sum of its path's
//    logits and Lam[d] = lse_1 + ... + lse_d.  L is carried as an unevaluated
//    float pair (hi + lo), in which sums of bf16/fp32 logits are exact, so two
//    paths of equal depth and equal logit sum get identical scores and the tie
//    rule decides between them; log rho itself is a float pair (~2^-44
//    relative), far inside the 1e-6 band where floating point may decide.
//  * Frontier: node p has one pending candidate, its next-ranked child (p, j);
//    with sorted ranks, the best of these is the best candidate overall.  The
//    pending candidate of node p is held in lane p % 32, register slot p / 32,
//    as a 96-bit key: order-preserving images of the hi and lo floats of log
//    rho, then tie bits 0xFFFFFF - (depth<<18 | rank<<8 | parent) so equal
//    scores prefer lower depth, rank and parent.  A pop is three redux.sync
//    reductions over the lanes' cached best keys.
//  * Each slot keeps, in a shared-memory record, its next-ranked candidate
//    (key and logit sum) and the first-child key of both its current and next
//    candidate.  A pop reads the winner's record: the winner's slot moves to
//    its next candidate and the new node's slot starts at the precomputed first
//    child, so the pop itself does only integer work and one expf (rho of the
//    winner, for the stop test).  The three records the pop invalidates are
//    recomputed afterwards, one per lane in a single SIMT pass.
//  * Stop test before adding candidate c to a tree of N nodes (C > 0):
//    S(N+1) < S(N)  <=>  rho_c C(N) < A_hat (C(N+1) - C(N)), in fp32 with
//    A_hat summed with Kahan compensation.
//  * Ancestor masks are built in shared memory and stored row by row.
#include "common.cuh"

namespace bastion {

namespace {

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

struct F2 {  // unevaluated sum hi + lo, |lo| <= ulp(hi)/2
  float h, l;
};

// a + b (float) with the rounding error of the leading sum kept (TwoSum).
__device__ __forceinline__ F2 f2_add(F2 a, float b) {
  const float s = a.h + b;
  if (!isfinite(s)) return {s, 0.f};
  const float bb = s - a.h;
  float e = (a.h - (s - bb)) + (b - bb);
  e += a.l;
  const float h = s + e;
  return {h, e - (h - s)};
}

// a - b for two pairs.
__device__ __forceinline__ F2 f2_sub(F2 a, F2 b) {
  const float s = a.h - b.h;
  if (!isfinite(s)) return {s, 0.f};
  const float bb = s - a.h;
  float e = (a.h - (s - bb)) + (-b.h - bb);
  e += a.l - b.l;
  const float h = s + e;
  return {h, e - (h - s)};
}

__device__ __forceinline__ bool key_gt(uint32_t ah, uint32_t al, uint32_t at, uint32_t bh,
                                       uint32_t bl, uint32_t bt) {
  if (ah != bh) return ah > bh;
  if (al != bl) return al > bl;
  return at > bt;
}

// Record of a candidate (parent P, rank j, depth d): its key, its logit sum and
// the key of its first child (whose parent index is filled in at pop time).
struct Cand {
  uint32_t h, l, t;    // key (0, 0, 0 = none)
  F2 L;                // path logit sum
  uint32_t ch, cl, ct; // first child key; ct lacks the child's parent index
};

__device__ __forceinline__ Cand cand_of(F2 Lp, int P, int d, int j, int b, int R, const float *lg,
                                        const F2 *Lam) {
  Cand c = {0u, 0u, 0u, {0.f, 0.f}, 0u, 0u, 0u};
  if (j >= R) return c;
  c.L = f2_add(Lp, lg[(d - 1) * R + j]);
  const F2 lr = f2_sub(c.L, Lam[d]);
  c.h = ord_f32(lr.h);
  c.l = ord_f32(lr.l);
  c.t = 0xFFFFFFu - (((uint32_t)d << 18) | ((uint32_t)j << 8) | (uint32_t)P);
  if (d < b) {
    const F2 lg2 = f2_sub(f2_add(c.L, lg[d * R]), Lam[d + 1]);
    c.ch = ord_f32(lg2.h);
    c.cl = ord_f32(lg2.l);
    c.ct = 0xFFFFFFu - ((uint32_t)(d + 1) << 18);
  }
  return c;
}

// Shared-memory record of slot s: its current candidate's logit sum and first
// child key, and its next candidate (key, logit sum, first child key).
struct Rec {
  F2 cL;
  uint32_t ch, cl, ct;
  uint32_t nh, nl, nt;
  F2 nL;
  uint32_t nch, ncl, nct;
  uint32_t pad[3];
};

template <int S>  // register slots per lane: S * 32 >= n_max
__global__ void __launch_bounds__(32) build_tree_kernel(TreeArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  Rec *rec = reinterpret_cast<Rec *>(smem);                         // [n_max]
  F2 *Lam = reinterpret_cast<F2 *>(rec + a.n_max);                  // [33]
  F2 *Lnode = Lam + 33;                                              // [n_max] node logit sums
  float *C = reinterpret_cast<float *>(Lnode + a.n_max);             // [n_max + 1]
  uint32_t *mask = reinterpret_cast<uint32_t *>(C + a.n_max + 1);   // [n_max * W]
  float *lg = reinterpret_cast<float *>(mask + a.n_max * a.W);      // [b * R]
  int *tk = reinterpret_cast<int *>(lg + a.b * a.R);                 // [b * R]

  const int r = blockIdx.x, lane = threadIdx.x;
  const int R = a.R, W = a.W, b = a.b;
  griddep_wait();
  griddep_launch_dependents();
  for (int idx = lane; idx < b * R; idx += 32) {
    const int d = idx / R, j = idx - d * R;
    lg[idx] = a.topk_logit[((size_t)r * b + d) * a.K + j];
    tk[idx] = a.topk_tok[((size_t)r * b + d) * a.K + j];
  }
  const float *cr = a.cost + (a.cost_per_request ? (size_t)r * (a.n_max + 1) : 0);
  bool bad = false;
  for (int i = lane; i <= a.n_max; i += 32) {
    const float c = cr[i];
    C[i] = c;
    if (i >= 1) bad |= !(c > 0.f) || isinf(c);
  }
  if (__any_sync(kFull, bad) && lane == 0) atomicOr(&a.status[r], BASTION_STATUS_BAD_COST);
  {
    // Lam[d] = lse_1 + ... + lse_d: each lse as a float pair, then a prefix scan
    F2 v = {0.f, 0.f};
    if (lane < b) {
      const double x = a.lse[(size_t)r * b + lane];
      const float h = (float)x;
      v = {h, (float)(x - (double)h)};
    }
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const F2 u = {__shfl_up_sync(kFull, v.h, o), __shfl_up_sync(kFull, v.l, o)};
      if (lane >= o) v = f2_sub(v, F2{-u.h, -u.l});
    }
    if (lane < b) Lam[lane + 1] = v;
    if (lane == 0) Lam[0] = {0.f, 0.f};
  }
  const int ctx = a.ctx_len[r];
  const float L_ar = a.l_ar[r];
  const size_t nb = (size_t)r * a.n_max;
  if (lane == 0) {
    a.parent[nb] = -1;
    a.depth[nb] = 0;
    a.pos_id[nb] = ctx;
    a.token[nb] = a.root_token[r];
    a.rank[nb] = -1;
    a.log_rho[nb] = 0.f;
    a.a_hat[nb] = 1.f;
    a.speedup[nb] = L_ar / C[1];
    Lnode[0] = {0.f, 0.f};
  }
  for (int w = lane; w < W; w += 32) {
    const uint32_t m = w == 0 ? 1u : 0u;
    mask[w] = m;
    a.anc_mask[nb * W + w] = m;
  }
  __syncwarp();

  // the root's slot: current candidate (0, 0), next (0, 1)
  uint32_t kh[S], kl[S], kt[S];
#pragma unroll
  for (int s = 0; s < S; ++s) kh[s] = kl[s] = kt[s] = 0u;
  {
    const Cand c = cand_of({0.f, 0.f}, 0, 1, lane, b, R, lg, Lam);  // lanes 0, 1 used
    const Cand c0 = {__shfl_sync(kFull, c.h, 0), __shfl_sync(kFull, c.l, 0), __shfl_sync(kFull, c.t, 0),
                     {__shfl_sync(kFull, c.L.h, 0), __shfl_sync(kFull, c.L.l, 0)},
                     __shfl_sync(kFull, c.ch, 0), __shfl_sync(kFull, c.cl, 0), __shfl_sync(kFull, c.ct, 0)};
    if (lane == 1) {
      Rec q;
      q.cL = c0.L; q.ch = c0.ch; q.cl = c0.cl; q.ct = c0.ct;
      q.nh = c.h; q.nl = c.l; q.nt = c.t; q.nL = c.L; q.nch = c.ch; q.ncl = c.cl; q.nct = c.ct;
      rec[0] = q;
    }
    if (lane == 0) { kh[0] = c0.h; kl[0] = c0.l; kt[0] = c0.t; }
  }
  __syncwarp();
  uint32_t bh = kh[0], bl = kl[0], bt = kt[0];

  float A_hi = 1.f, A_lo = 0.f;  // A_hat with Kahan compensation
  int N = 1;
  while (N < a.n_max) {
    const uint32_t mh = __reduce_max_sync(kFull, bh);
    const uint32_t ml = __reduce_max_sync(kFull, bh == mh ? bl : 0u);
    const uint32_t mt = __reduce_max_sync(kFull, (bh == mh && bl == ml) ? bt : 0u);
    if ((mh | ml | mt) == 0u) break;  // no candidate left
    const float lr_h = unord_f32(mh), lr_l = unord_f32(ml);
    if (lr_h == -INFINITY) break;
    const uint32_t sec = 0xFFFFFFu - mt;
    const int d = (int)(sec >> 18), j = (int)((sec >> 8) & 1023u), p = (int)(sec & 255u);
    const float e = lr_h < -104.f ? 0.f : expf(lr_h);
    const float rho = fmaf(e, lr_l, e);
    const float Cp = C[N], Cn = C[N + 1];
    if (rho * Cp < (A_hi + A_lo) * (Cn - Cp)) break;  // S would decrease: keep T_N

    const int n = N;
    N = n + 1;
    {
      const float y = rho - A_lo;
      const float t = A_hi + y;
      A_lo = (t - A_hi) - y;
      A_hi = t;
    }
    const Rec w = rec[p];
    // critical path: the two slots that change
    if (lane == (p & 31)) {
      const int s0 = p >> 5;
#pragma unroll
      for (int s = 0; s < S; ++s)
        if (s == s0) { kh[s] = w.nh; kl[s] = w.nl; kt[s] = w.nt; }
    }
    if (d < b && lane == (n & 31)) {
      const int s1 = n >> 5;
#pragma unroll
      for (int s = 0; s < S; ++s)
        if (s == s1) { kh[s] = w.ch; kl[s] = w.cl; kt[s] = w.ct - (uint32_t)n; }
    }
    if (lane == (p & 31) || (d < b && lane == (n & 31))) {
      bh = kh[0]; bl = kl[0]; bt = kt[0];
#pragma unroll
      for (int s = 1; s < S; ++s)
        if (key_gt(kh[s], kl[s], kt[s], bh, bl, bt)) { bh = kh[s]; bl = kl[s]; bt = kt[s]; }
    }
    // the records this pop invalidates, one per lane:
    //   lane 0: slot p's new next candidate (p, j + 2)
    //   lane 1: the new node's current candidate (n, 0) (logit sum, first child)
    //   lane 2: the new node's next candidate (n, 1)
    {
      F2 Lpar = w.cL;  // the new node's logit sum
      int P = n, dd = d + 1, jj = lane - 1;
      if (lane == 0) { Lpar = Lnode[p]; P = p; dd = d; jj = j + 2; }
      Cand c = {0u, 0u, 0u, {0.f, 0.f}, 0u, 0u, 0u};
      if (lane < 3 && dd <= b) c = cand_of(Lpar, P, dd, jj, b, R, lg, Lam);
      __syncwarp();
      if (lane == 3) Lnode[n] = w.cL;
      if (lane == 0) {
        // slot p advances: current <- next, next <- (p, j + 2)
        Rec q = w;
        q.cL = w.nL; q.ch = w.nch; q.cl = w.ncl; q.ct = w.nct;
        q.nh = c.h; q.nl = c.l; q.nt = c.t; q.nL = c.L; q.nch = c.ch; q.ncl = c.cl; q.nct = c.ct;
        rec[p] = q;
      }
      if (d < b) {
        if (lane == 1) { rec[n].cL = c.L; rec[n].ch = c.ch; rec[n].cl = c.cl; rec[n].ct = c.ct; }
        if (lane == 2) {
          rec[n].nh = c.h; rec[n].nl = c.l; rec[n].nt = c.t; rec[n].nL = c.L;
          rec[n].nch = c.ch; rec[n].ncl = c.cl; rec[n].nct = c.ct;
        }
      }
    }
    if (lane == 0) {
      const size_t o = nb + n;
      const float Ah = A_hi + A_lo;
      a.parent[o] = p;
      a.depth[o] = d;
      a.pos_id[o] = ctx + d;
      a.token[o] = tk[(d - 1) * R + j];
      a.rank[o] = j;
      a.log_rho[o] = lr_h;
      a.a_hat[o] = Ah;
      a.speedup[o] = Ah * L_ar / Cn;
    }
    for (int q = lane; q < W; q += 32) {
      const uint32_t m = mask[p * W + q] | (q == (n >> 5) ? (1u << (n & 31)) : 0u);
      mask[n * W + q] = m;
      a.anc_mask[(nb + n) * W + q] = m;
    }
    __syncwarp();
  }
  if (lane == 0) a.n_nodes[r] = N;
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
  const size_t smem = (size_t)n_max * 64 + 33 * 8 + (size_t)n_max * 8 + (size_t)(n_max + 1) * 4 +
                      (size_t)n_max * a.W * 4 + (size_t)b * a.R * 8;
  if (n_max <= 32) launch_s<1>(a, smem, stream);
  else if (n_max <= 64) launch_s<2>(a, smem, stream);
  else if (n_max <= 128) launch_s<4>(a, smem, stream);
  else launch_s<8>(a, smem, stream);
  return cudaGetLastError() == cudaSuccess ? BASTION_OK : BASTION_ERR_LAUNCH;
}

}  // namespace bastion
