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
//  * Each slot keeps, in a shared-memory record, its current and next-ranked
//    candidates (logit sum, rho, first-child key; the next one's key too).  A
//    pop reads the winner's record: the winner's slot moves to its next
//    candidate and the new node's slot starts at the precomputed first child,
//    so the pop itself does only integer work and selects.  The three records
//    the pop invalidates are recomputed one per lane in the same straight-line
//    block as the next pop's reductions, so the two overlap.
//  * Stop test before adding candidate c to a tree of N nodes (C > 0):
//    S(N+1) < S(N)  <=>  rho_c C(N) < A_hat (C(N+1) - C(N)), in fp32 with
//    A_hat summed with Kahan compensation.
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

struct F2 {  // unevaluated sum hi + lo, |lo| <= ulp(hi)/2
  float h, l;
};

// a + b (float) with the rounding error of the leading sum kept (TwoSum);
// a non-finite leading sum is returned as (sum, 0).
__device__ __forceinline__ F2 f2_add(F2 a, float b) {
  const float s = a.h + b;
  const float bb = s - a.h;
  float e = (a.h - (s - bb)) + (b - bb);
  e += a.l;
  const float h = s + e;
  const float l = e - (h - s);
  const bool fin = isfinite(s);
  return {fin ? h : s, fin ? l : 0.f};
}

// a - b for two pairs.
__device__ __forceinline__ F2 f2_sub(F2 a, F2 b) {
  const float s = a.h - b.h;
  const float bb = s - a.h;
  float e = (a.h - (s - bb)) + (-b.h - bb);
  e += a.l - b.l;
  const float h = s + e;
  const float l = e - (h - s);
  const bool fin = isfinite(s);
  return {fin ? h : s, fin ? l : 0.f};
}

// 96-bit key comparison a > b without branches.
__device__ __forceinline__ bool key_gt(uint32_t ah, uint32_t al, uint32_t at, uint32_t bh,
                                       uint32_t bl, uint32_t bt) {
  return (ah > bh) | ((ah == bh) & ((al > bl) | ((al == bl) & (at > bt))));
}

// rho of a candidate from its log rho pair (0 below the float range).
__device__ __forceinline__ float rho_of(F2 lr) {
  const float e = lr.h < -104.f ? 0.f : expf(lr.h);
  return fmaf(e, lr.l, e);
}

// A candidate (parent P, rank j, depth d): its key, logit sum, rho and the
// key of its first child (whose parent index is filled in at pop time).
struct Cand {
  uint32_t h, l, t;    // key (0, 0, 0 = none)
  F2 L;                // path logit sum
  float rho;
  uint32_t ch, cl, ct; // first child key; ct lacks the child's parent index
};

// Branch-free: invalid (or out of range) candidates come back as key 0.
__device__ __forceinline__ Cand cand_of(F2 Lp, int P, int d, int j, bool valid, int b, int R,
                                        const float *lg, const F2 *Lam) {
  valid = valid && j < R && d >= 1 && d <= b;
  const int jj = valid ? j : 0, dd = valid ? d : 1;
  Cand c;
  c.L = f2_add(Lp, lg[(dd - 1) * R + jj]);
  const F2 lr = f2_sub(c.L, Lam[dd]);
  c.h = valid ? ord_f32(lr.h) : 0u;
  c.l = valid ? ord_f32(lr.l) : 0u;
  c.t = valid ? 0xFFFFFFu - (((uint32_t)dd << 18) | ((uint32_t)jj << 8) | (uint32_t)P) : 0u;
  c.rho = rho_of(lr);
  const bool kid = valid && dd < b;
  const int dc = dd < b ? dd : b - 1;  // a valid row to read either way
  const F2 lg2 = f2_sub(f2_add(c.L, lg[dc * R]), Lam[dc + 1]);
  c.ch = kid ? ord_f32(lg2.h) : 0u;
  c.cl = kid ? ord_f32(lg2.l) : 0u;
  c.ct = kid ? 0xFFFFFFu - ((uint32_t)(dd + 1) << 18) : 0u;
  return c;
}

// Shared-memory record of slot s: its current candidate (logit sum, rho,
// first child key) and its next candidate (key, rho, logit sum, first child
// key).
struct __align__(16) Rec {
  F2 cL;
  uint32_t ch, cl, ct;
  float crho;
  uint32_t nh, nl, nt;
  float nrho;
  F2 nL;
  uint32_t nch, ncl, nct;
  uint32_t pad;
};

template <int S>  // register slots per lane: S * 32 >= n_max
__global__ void __launch_bounds__(32) build_tree_kernel(TreeArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  Rec *rec = reinterpret_cast<Rec *>(smem);                         // [n_max]
  float *lg = reinterpret_cast<float *>(rec + a.n_max);              // [b * R] (16-byte aligned)
  int *tk = reinterpret_cast<int *>(lg + a.b * a.R);                 // [b * R]
  F2 *Lam = reinterpret_cast<F2 *>(tk + a.b * a.R);                  // [33]
  F2 *Lnode = Lam + 33;                                              // [n_max] node logit sums
  float *C = reinterpret_cast<float *>(Lnode + a.n_max);             // [n_max + 1]
  uint32_t *mask = reinterpret_cast<uint32_t *>(C + a.n_max + 1);   // [n_max * W]
  int *nd_par = reinterpret_cast<int *>(mask + a.n_max * a.W);       // [n_max] per node:
  int *nd_dj = nd_par + a.n_max;                                     //   depth << 16 | rank
  float *nd_lr = reinterpret_cast<float *>(nd_dj + a.n_max);         //   log rho (hi)
  float *nd_A = nd_lr + a.n_max;                                     //   A_hat after it

  const int r = blockIdx.x, lane = threadIdx.x;
  const int R = a.R, W = a.W, b = a.b;
  griddep_wait();
  griddep_launch_dependents();
  // ---- stage the request's inputs; every load of a batch is issued before use
  const int ctx = a.ctx_len[r];
  const float L_ar = a.l_ar[r];
  const int root_tok = a.root_token[r];
  const double lse_v = lane < b ? a.lse[(size_t)r * b + lane] : 0.0;
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
    const bool vec = R == a.K && (nlg & 3) == 0 && ((uintptr_t)gl & 15) == 0 &&
                     ((uintptr_t)gt & 15) == 0;
    if (vec) {  // the [b][K] block is contiguous: 16-byte loads
      const int n4 = nlg >> 2;
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
          if (i < n4) {
            reinterpret_cast<float4 *>(lg)[i] = v[u];
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
          if (idx < nlg) {
            lg[idx] = v[u];
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
  {
    // Lam[d] = lse_1 + ... + lse_d: each lse as a float pair, then a prefix scan
    F2 v = {0.f, 0.f};
    if (lane < b) {
      const float h = (float)lse_v;
      v = {h, (float)(lse_v - (double)h)};
    }
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const F2 u = {__shfl_up_sync(kFull, v.h, o), __shfl_up_sync(kFull, v.l, o)};
      if (lane >= o) v = f2_sub(v, F2{-u.h, -u.l});
    }
    if (lane < b) Lam[lane + 1] = v;
    if (lane == 0) Lam[0] = {0.f, 0.f};
  }
  if (lane == 0) Lnode[0] = {0.f, 0.f};
  for (int w = lane; w < W; w += 32) mask[w] = w == 0 ? 1u : 0u;
  __syncwarp();

  // the root's slot: current candidate (0, 0), next (0, 1)
  uint32_t kh[S], kl[S], kt[S];
#pragma unroll
  for (int s = 0; s < S; ++s) kh[s] = kl[s] = kt[s] = 0u;
  {
    const Cand c = cand_of({0.f, 0.f}, 0, 1, lane, lane < 2, b, R, lg, Lam);  // lanes 0, 1
    const float c0rho = __shfl_sync(kFull, c.rho, 0);
    const F2 c0L = {__shfl_sync(kFull, c.L.h, 0), __shfl_sync(kFull, c.L.l, 0)};
    const uint32_t c0ch = __shfl_sync(kFull, c.ch, 0), c0cl = __shfl_sync(kFull, c.cl, 0),
                   c0ct = __shfl_sync(kFull, c.ct, 0);
    if (lane == 1) {
      Rec q;
      q.cL = c0L; q.ch = c0ch; q.cl = c0cl; q.ct = c0ct; q.crho = c0rho;
      q.nh = c.h; q.nl = c.l; q.nt = c.t; q.nrho = c.rho; q.nL = c.L;
      q.nch = c.ch; q.ncl = c.cl; q.nct = c.ct; q.pad = 0u;
      rec[0] = q;
    }
    if (lane == 0) { kh[0] = c.h; kl[0] = c.l; kt[0] = c.t; }
  }
  __syncwarp();
  uint32_t bh = kh[0], bl = kl[0], bt = kt[0];
  uint32_t mh = __reduce_max_sync(kFull, bh);
  uint32_t ml = __reduce_max_sync(kFull, bh == mh ? bl : 0u);
  uint32_t mt = __reduce_max_sync(kFull, (bh == mh && bl == ml) ? bt : 0u);

  float A_hi = 1.f, A_lo = 0.f;  // A_hat with Kahan compensation
  int N = 1;
  while (N < a.n_max) {
    if ((mh | ml | mt) == 0u) break;  // no candidate left
    const float lr_h = unord_f32(mh);
    if (lr_h == -INFINITY) break;
    const uint32_t sec = 0xFFFFFFu - mt;
    const int d = (int)(sec >> 18), j = (int)((sec >> 8) & 1023u), p = (int)(sec & 255u);
    const Rec w = rec[p];
    const float Cp = C[N], Cn = C[N + 1];
    if (w.crho * Cp < (A_hi + A_lo) * (Cn - Cp)) break;  // S would decrease: keep T_N

    const int n = N;
    N = n + 1;
    {
      const float y = w.crho - A_lo;
      const float t = A_hi + y;
      A_lo = (t - A_hi) - y;
      A_hi = t;
    }
    // the two slots that change: p moves to its next candidate, n starts at its
    // first child; then every lane rescans its slots
    const bool kid = d < b;
    const int lp = p & 31, sp = p >> 5, ln = n & 31, sn = n >> 5;
#pragma unroll
    for (int s = 0; s < S; ++s) {
      const bool up = lane == lp && s == sp;
      const bool un = kid && lane == ln && s == sn;
      kh[s] = up ? w.nh : (un ? w.ch : kh[s]);
      kl[s] = up ? w.nl : (un ? w.cl : kl[s]);
      kt[s] = up ? w.nt : (un ? w.ct - (uint32_t)n : kt[s]);
    }
    bh = kh[0]; bl = kl[0]; bt = kt[0];
#pragma unroll
    for (int s = 1; s < S; ++s) {
      const bool g = key_gt(kh[s], kl[s], kt[s], bh, bl, bt);
      bh = g ? kh[s] : bh; bl = g ? kl[s] : bl; bt = g ? kt[s] : bt;
    }
    // the records this pop invalidates, one per lane, and the next pop's
    // reductions (independent of them):
    //   lane 0: slot p's new next candidate (p, j + 2)
    //   lane 1: the new node's current candidate (n, 0)
    //   lane 2: the new node's next candidate (n, 1)
    const bool l0 = lane == 0;
    const F2 Lpar = l0 ? Lnode[p] : w.cL;
    const Cand c = cand_of(Lpar, l0 ? p : n, l0 ? d : d + 1, l0 ? j + 2 : lane - 1,
                           l0 || (kid && lane < 3), b, R, lg, Lam);
    mh = __reduce_max_sync(kFull, bh);
    ml = __reduce_max_sync(kFull, bh == mh ? bl : 0u);
    mt = __reduce_max_sync(kFull, (bh == mh && bl == ml) ? bt : 0u);
    if (l0) {  // slot p advances: current <- next, next <- (p, j + 2)
      Rec q;
      q.cL = w.nL; q.ch = w.nch; q.cl = w.ncl; q.ct = w.nct; q.crho = w.nrho;
      q.nh = c.h; q.nl = c.l; q.nt = c.t; q.nrho = c.rho; q.nL = c.L;
      q.nch = c.ch; q.ncl = c.cl; q.nct = c.ct; q.pad = 0u;
      rec[p] = q;
    }
    if (kid && lane == 1) {
      rec[n].cL = c.L; rec[n].ch = c.ch; rec[n].cl = c.cl; rec[n].ct = c.ct; rec[n].crho = c.rho;
    }
    if (kid && lane == 2) {
      rec[n].nh = c.h; rec[n].nl = c.l; rec[n].nt = c.t; rec[n].nrho = c.rho; rec[n].nL = c.L;
      rec[n].nch = c.ch; rec[n].ncl = c.cl; rec[n].nct = c.ct;
    }
    if (lane == 3) Lnode[n] = w.cL;
    if (lane == 4) {
      nd_par[n] = p;
      nd_dj[n] = (d << 16) | j;
      nd_lr[n] = lr_h;
      nd_A[n] = A_hi + A_lo;
    }
    if (lane < W) mask[n * W + lane] = mask[p * W + lane] | (lane == (n >> 5) ? (1u << (n & 31)) : 0u);
    __syncwarp();
  }

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
      a.log_rho[o] = nd_lr[i];
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
  const size_t smem = (size_t)n_max * sizeof(Rec) + 33 * 8 + (size_t)n_max * 8 +
                      (size_t)(n_max + 1) * 4 + (size_t)n_max * a.W * 4 + (size_t)b * a.R * 8 +
                      (size_t)n_max * 16;
  if (n_max <= 32) launch_s<1>(a, smem, stream);
  else if (n_max <= 64) launch_s<2>(a, smem, stream);
  else if (n_max <= 128) launch_s<4>(a, smem, stream);
  else launch_s<8>(a, smem, stream);
  return cudaGetLastError() == cudaSuccess ? BASTION_OK : BASTION_ERR_LAUNCH;
}

}  // namespace bastion
