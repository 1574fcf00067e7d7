// Steps 2-3 of the draft-tree path as device code: staging a request's
// tables, the best-first pops, and the tree's outputs.
//
// Bastion (gist.science/nl/paper/2605.29727), Methodologie §1 ("Pad-scoren":
// rho(i) = prod_{k<=d(i)} q_k(x_ik)), §2 ("Surrogaat-schatting": A_hat = sum rho;
// "Optimale Constructie": add the valid node with the highest rho), §3
// ("Adaptief Stoppen": grow until S(N) = A_hat(T_N) L_AR / C(N) starts to fall).
//
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
//  * The request's tables are staged into shared memory by the CTA's four
//    warps, with several loads in flight per thread; then warps 1-3 leave and
//    warp 0 runs the pops alone (a warp whose CTA has other warps parked at a
//    barrier ran the same pops about three times slower) and writes the
//    per-node results and ancestor masks out, coalesced.
#pragma once

#include "common.cuh"

namespace bastion {

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

namespace tb {

constexpr float kFix = 1099511627776.f;         // 2^40
constexpr float kUnfix = 9.094947017729282e-13f;  // 2^-40
constexpr int64_t kNegFix = -(1ll << 58);         // the score of a -inf logit
constexpr int64_t kInfCut = -(1ll << 57);         // scores below count as -inf
constexpr float kMaxLogit = 131072.f;             // finite logits clamped to 2^17

// Fixed-point images (2^-40 units) of a logit and of an lse value.
__device__ __forceinline__ int64_t fix_logit(float x) {
  if (!(x > -INFINITY)) return kNegFix;  // -inf (and NaN, which the top-K step flags)
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

// rho = exp(score 2^-40).  x = k ln 2 + f with k the nearest integer to x / ln 2
// (from an estimate of x within 2^-8, the top 32 bits) and f = score - k ln 2
// exact in fixed point (|f| < 0.36), then 2^k expf(f) with f rounded to 2^-31:
// within 2.2 2^-23 (relative) of exact, using 32-bit converts only (a
// conversion between a 64-bit integer and a float costs ~100 cycles here, and
// the next pop's stop test waits on this value through A_hat).
constexpr int64_t kLn2Fix = 762123384786ll;  // ln 2 in 2^-40 units, rounded
__device__ __forceinline__ float rho_of(int64_t score) {
  const int64_t D = score < -(104ll << 40) ? -(104ll << 40) : score;
  const float xa = (float)(int)(D >> 32) * 0.00390625f;
  const int k = __float2int_rn(xa * 1.4426950408889634f);
  const int64_t f = D - (int64_t)k * kLn2Fix;
  const float ff = (float)(int)(f >> 9) * 4.656612873077393e-10f;
  const float r = ldexpf(expf(ff), k);
  return score < -(104ll << 40) ? 0.f : r;
}

// The largest 96-bit key over the warp.
__device__ __forceinline__ void warp_best(uint32_t bh, uint32_t bl, uint32_t bt, uint32_t &mh,
                                          uint32_t &ml, uint32_t &mt) {
  mh = __reduce_max_sync(kFull, bh);
  ml = __reduce_max_sync(kFull, bh == mh ? bl : 0u);
  mt = __reduce_max_sync(kFull, (bh == mh && bl == ml) ? bt : 0u);
}


// Shared-memory layout of one request's build.
struct TreeSmem {
  int64_t *nd_sc;   // [n_max] node scores (first, padded to an even count)
  int64_t *lq;      // [b * R] the scores' steps
  int *tk;          // [b * R] tokens
  float *C;         // [n_max + 1]
  uint32_t *mask;   // [n_max * W]
  int *nd_par;      // [n_max]
  int *nd_dj;       // [n_max] depth << 16 | rank
  float *nd_A;      // [n_max] A_hat after the node
  int *misc;        // [4]: misc[0] = the tree size N
};

__host__ __device__ inline size_t tree_smem_bytes(int b, int R, int n_max, int W) {
  return (size_t)((n_max + 1) & ~1) * 8 + (size_t)b * R * 12 + (size_t)(n_max + 1) * 4 +
         (size_t)n_max * W * 4 + (size_t)n_max * 12 + 16;
}

__device__ __forceinline__ TreeSmem tree_smem(unsigned char *base, const TreeArgs &a) {
  TreeSmem t;
  t.nd_sc = reinterpret_cast<int64_t *>(base);
  t.lq = t.nd_sc + ((a.n_max + 1) & ~1);
  t.tk = reinterpret_cast<int *>(t.lq + a.b * a.R);
  t.C = reinterpret_cast<float *>(t.tk + a.b * a.R);
  t.mask = reinterpret_cast<uint32_t *>(t.C + a.n_max + 1);
  t.nd_par = reinterpret_cast<int *>(t.mask + a.n_max * a.W);
  t.nd_dj = t.nd_par + a.n_max;
  t.nd_A = reinterpret_cast<float *>(t.nd_dj + a.n_max);
  t.misc = reinterpret_cast<int *>(t.nd_A + a.n_max);
  return t;
}

// Stages request r's tables (nt threads of the CTA, thread index tid; the
// caller synchronises the CTA afterwards).  Returns true on a thread that saw
// a cost entry C(N), N >= 1, that is not finite and positive.
__device__ __forceinline__ bool stage_request(const TreeArgs &a, int r, const TreeSmem &t, int tid,
                                              int nt) {
  const int R = a.R, b = a.b;
  const int nlg = b * R;
  // the cost row's loads are issued first and used last, so they travel with
  // the tables' (the cost table is never written by this grid)
  const float *cr = a.cost + (a.cost_per_request ? (size_t)r * (a.n_max + 1) : 0);
  constexpr int kCv = 3;
  float cv[kCv];
#pragma unroll
  for (int k = 0; k < kCv; ++k) {
    const int i = tid + k * nt;
    cv[k] = i <= a.n_max ? __ldg(cr + i) : 1.f;
  }
  const float *gl = a.topk_logit + (size_t)r * b * a.K;
  const int32_t *gt = a.topk_tok + (size_t)r * b * a.K;
  const double *gs = a.lse + (size_t)r * b;
  const bool vec = R == a.K && (R & 3) == 0 && ((uintptr_t)gl & 15) == 0 && ((uintptr_t)gt & 15) == 0;
  constexpr int U = 4;  // loads in flight per thread before any is used
  if (vec) {  // the [b][K] block is contiguous and each 16 bytes lie in one row
    const int n4 = nlg >> 2, r4 = R >> 2;
    for (int i0 = tid; i0 < n4; i0 += nt * U) {
      float4 v[U];
      int4 tv[U];
      double ls[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = i0 + u * nt;
        if (i < n4) {
          v[u] = __ldg(reinterpret_cast<const float4 *>(gl) + i);
          tv[u] = __ldg(reinterpret_cast<const int4 *>(gt) + i);
          ls[u] = __ldg(gs + i / r4);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = i0 + u * nt;
        if (i < n4) {
          const int64_t lf = fix_lse(ls[u]);
          const float e[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int64_t f = fix_logit(e[q]);
            t.lq[4 * i + q] = f == kNegFix ? kNegFix : f - lf;
          }
          reinterpret_cast<int4 *>(t.tk)[i] = tv[u];
        }
      }
    }
  } else {
    for (int i0 = tid; i0 < nlg; i0 += nt * U) {
      float v[U];
      int tv[U];
      double ls[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int idx = i0 + u * nt;
        if (idx < nlg) {
          const int d = idx / R, j = idx - d * R;
          v[u] = __ldg(gl + (size_t)d * a.K + j);
          tv[u] = __ldg(gt + (size_t)d * a.K + j);
          ls[u] = __ldg(gs + d);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int idx = i0 + u * nt;
        if (idx < nlg) {
          const int64_t f = fix_logit(v[u]);
          t.lq[idx] = f == kNegFix ? kNegFix : f - fix_lse(ls[u]);
          t.tk[idx] = tv[u];
        }
      }
    }
  }
  bool bad = false;
#pragma unroll
  for (int k = 0; k < kCv; ++k) {
    const int i = tid + k * nt;
    if (i <= a.n_max) {
      t.C[i] = cv[k];
      if (i >= 1) bad |= !(cv[k] > 0.f) || isinf(cv[k]);
    }
  }
  for (int i = tid + kCv * nt; i <= a.n_max; i += nt) {
    const float c = __ldg(cr + i);
    t.C[i] = c;
    bad |= !(c > 0.f) || isinf(c);
  }
  for (int w = tid; w < a.W; w += nt) t.mask[w] = w == 0 ? 1u : 0u;
  return bad;
}

// Warp 0's build of the staged request; returns the tree size N (also in
// t.misc[0]).  S register slots per lane (S * 32 >= n_max).
template <int S>
__device__ __forceinline__ int pop_all(const TreeArgs &a, const TreeSmem &t, int lane) {
  const int R = a.R, W = a.W, b = a.b;
  uint32_t kh[S], kl[S], kt[S];
  int64_t sc[S];
#pragma unroll
  for (int s = 0; s < S; ++s) { kh[s] = kl[s] = kt[s] = 0u; sc[s] = 0; }
  if (lane == 0) {  // the root: score 0, pending candidate (0, 0) at depth 1
    const uint64_t k = key_of(t.lq[0]);
    kh[0] = (uint32_t)(k >> 32);
    kl[0] = (uint32_t)k;
    kt[0] = 0xFFFFFFu - (1u << 18);
  }
  uint32_t mh, ml, mt;
  warp_best(kh[0], kl[0], kt[0], mh, ml, mt);
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
    const int64_t qs = t.lq[(d - 1) * R + (vs ? jn : j)];
    const int64_t qc = t.lq[(vc ? d : d - 1) * R];
    const uint32_t mrow = lane < W ? t.mask[p * W + lane] : 0u;
    const float Cp = t.C[N], Cn = t.C[N + 1];
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
    uint32_t bh = kh[0], bl = kl[0], bt = kt[0];
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
      const float tt = A_hi + y;
      A_lo = (tt - A_hi) - y;
      A_hi = tt;
    }
    if (lane == 0) {
      t.nd_par[n] = p;
      t.nd_dj[n] = (d << 16) | j;
      t.nd_sc[n] = lr;
      t.nd_A[n] = A_hi + A_lo;
    }
    if (lane < W) t.mask[n * W + lane] = mrow | (lane == (n >> 5) ? (1u << (n & 31)) : 0u);
  }
  if (lane == 0) t.misc[0] = N;
  return N;
}

// The tree's outputs for request r, written by nt threads (after a CTA
// barrier that follows the pops).
__device__ __forceinline__ void write_tree(const TreeArgs &a, int r, const TreeSmem &t, int N,
                                           bool bad_cost, int tid, int nt) {
  const size_t nb = (size_t)r * a.n_max;
  const int R = a.R, W = a.W;
  const int ctx = a.ctx_len[r];
  const float L_ar = a.l_ar[r];
  if (tid == 0) {
    a.n_nodes[r] = N;
    if (bad_cost) atomicOr(&a.status[r], BASTION_STATUS_BAD_COST);
  }
  for (int i = tid; i < N; i += nt) {
    const size_t o = nb + i;
    if (i == 0) {
      a.parent[o] = -1;
      a.depth[o] = 0;
      a.pos_id[o] = ctx;
      a.token[o] = a.root_token[r];
      a.rank[o] = -1;
      a.log_rho[o] = 0.f;
      a.a_hat[o] = 1.f;
      a.speedup[o] = L_ar / t.C[1];
    } else {
      const int dj = t.nd_dj[i], d = dj >> 16, j = dj & 0xffff;
      const float Ah = t.nd_A[i];
      a.parent[o] = t.nd_par[i];
      a.depth[o] = d;
      a.pos_id[o] = ctx + d;
      a.token[o] = t.tk[(d - 1) * R + j];
      a.rank[o] = j;
      a.log_rho[o] = __ll2float_rn(t.nd_sc[i]) * kUnfix;
      a.a_hat[o] = Ah;
      a.speedup[o] = Ah * L_ar / t.C[i + 1];
    }
  }
  for (int q = tid; q < N * W; q += nt) a.anc_mask[nb * W + q] = t.mask[q];
}

inline TreeArgs tree_args(const float *topk_logit, const int32_t *topk_tok, const double *lse, int B,
                          int b, int K, int n_max, const int32_t *root_token, const int32_t *ctx_len,
                          const float *cost_ms, int cost_per_request, const float *l_ar,
                          int32_t *n_nodes, int32_t *parent, int32_t *depth, int32_t *pos_id,
                          int32_t *token, int32_t *rank, float *log_rho, float *a_hat, float *speedup,
                          uint32_t *anc_mask, int32_t *status) {
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
  return a;
}

// Register slots a lane needs for n_max nodes.
__host__ __device__ inline int tree_slots(int n_max) {
  return n_max <= 32 ? 1 : n_max <= 64 ? 2 : n_max <= 128 ? 4 : 8;
}

}  // namespace tb
}  // namespace bastion
