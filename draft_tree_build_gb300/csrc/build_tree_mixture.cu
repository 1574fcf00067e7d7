// Best-first draft trees on a latent-mixture proposal.
//
// DBlast ("Dependent Block Drafting", "Methodologie" 1, "Afhankelijke
// Blok-sampling via Latente Mix") writes the block proposal as a mixture over
// a latent branch z:  q_dep(x_1..b | y) = sum_z q(z|y) prod_i q_i(x_i | y, z).
// The tree of Bastion (gist.science/nl/paper/2605.29727, Methodologie §1-§3)
// is grown on the prefix score this induces, the mixture probability
//   rho(x_1..d) = sum_z pi_z prod_{k<=d} q_k^z(x_k),   pi_z = q(z|y),
// with the same controller: add the best candidate while S(N) = A_hat L_AR /
// C(N) does not decrease.  rho is non-increasing along a path, so best-first
// on it is exact, as in the single-proposal tree.
//
// Inputs per request: each branch's K ranked tokens per block position (the
// top-K step run per branch: logits, tokens, lse) and the branch weights pi.
// A token outside branch z's list at position k has q_k^z = 0; the children of
// a depth-d node are the union over z of the branches' tokens at position d+1.
//
// One warp builds one request's tree (requests are independent CTAs); this is
// the parity form of the step, in fp64 throughout:
//  * per position d, the union U_d of the branches' tokens is tabulated once,
//    with each branch's logit for each union token (-inf where absent);
//  * node n keeps, per branch, the sum of its path's logits (fp64) and one
//    pending candidate, its best untaken child under (log rho descending,
//    token ascending); a child's log rho is log sum_z exp(log pi_z + (logit
//    sum - lse sum)), with the largest term factored out;
//  * a pop takes the best pending candidate over the nodes under (log rho
//    descending, depth, token, parent ascending), runs the stop test
//    (A_hat + rho) L / C(N+1) < A_hat L / C(N), and then rescans two child
//    lists with warp-parallel argmaxes: the parent's (its next-best untaken
//    child) and the new node's.
// There is no wait of any kind: every loop is bounded by the tree budget or
// a table size.
#include <cmath>

#include "common.cuh"

namespace bastion {

namespace {

struct MixArgs {
  const float *topk_logit;  // [B, Z, b, K]
  const int32_t *topk_tok;  // [B, Z, b, K]
  const double *lse;        // [B, Z, b]
  const double *pi;         // [B, Z]
  int B, Z, b, K, n_max, W, E, UW;
  const int32_t *root_token, *ctx_len;
  const float *cost;
  int cost_per_request;
  const float *l_ar;
  int32_t *n_nodes, *parent, *depth, *pos_id, *token;
  float *log_rho, *a_hat, *speedup;
  uint32_t *anc_mask;
  int32_t *status;
};

// Shared-memory layout for one request (fp64 arrays first, 8-byte aligned).
struct MixLayout {
  size_t lam, lpi, ls, plr, lr;                       // double
  size_t ulg, utok, nu, cost, par, dep, tok, ah, sp;  // 4-byte
  size_t ptok, pu, mask, taken, etok, efirst, umap;
  size_t bytes;
};

__host__ __device__ inline MixLayout mix_layout(int Z, int b, int E, int n_max, int W, int UW) {
  MixLayout l;
  size_t o = 0;
  auto take = [&](size_t n) { const size_t at = o; o += n; return at; };
  l.lam = take((size_t)Z * (b + 1) * 8);
  l.lpi = take((size_t)Z * 8);
  l.ls = take((size_t)n_max * Z * 8);
  l.plr = take((size_t)n_max * 8);
  l.lr = take((size_t)n_max * 8);
  l.ulg = take((size_t)b * E * Z * 4);
  l.utok = take((size_t)b * E * 4);
  l.nu = take((size_t)b * 4);
  l.cost = take((size_t)(n_max + 1) * 4);
  l.par = take((size_t)n_max * 4);
  l.dep = take((size_t)n_max * 4);
  l.tok = take((size_t)n_max * 4);
  l.ah = take((size_t)n_max * 4);
  l.sp = take((size_t)n_max * 4);
  l.ptok = take((size_t)n_max * 4);
  l.pu = take((size_t)n_max * 4);
  l.mask = take((size_t)n_max * W * 4);
  l.taken = take((size_t)n_max * UW * 4);
  l.etok = take((size_t)E * 4);
  l.efirst = take((size_t)E * 4);
  l.umap = take((size_t)E * 4);
  l.bytes = o;
  return l;
}

constexpr double kNegInf = -INFINITY;

// (score, depth, token, node) order: true when a is better than b.
__device__ __forceinline__ bool mix_better(double sa, int da, int ta, int na, double sb, int db,
                                           int tb, int nb) {
  if (sa != sb) return sa > sb;
  if (da != db) return da < db;
  if (ta != tb) return ta < tb;
  return na < nb;
}

__global__ void __launch_bounds__(32) build_tree_mixture_kernel(MixArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int r = blockIdx.x, lane = threadIdx.x;
  const int Z = a.Z, b = a.b, K = a.K, E = a.E, n_max = a.n_max, W = a.W, UW = a.UW;
  const MixLayout L = mix_layout(Z, b, E, n_max, W, UW);
  double *Lam = reinterpret_cast<double *>(smem + L.lam);  // [Z][b+1]
  double *lpi = reinterpret_cast<double *>(smem + L.lpi);  // [Z]
  double *Ls = reinterpret_cast<double *>(smem + L.ls);    // [n_max][Z] logit sums
  double *plr = reinterpret_cast<double *>(smem + L.plr);  // [n_max] pending log rho
  double *lr = reinterpret_cast<double *>(smem + L.lr);    // [n_max] node log rho
  float *ulg = reinterpret_cast<float *>(smem + L.ulg);    // [b][E][Z] branch logits of U_d
  int *utok = reinterpret_cast<int *>(smem + L.utok);      // [b][E] tokens of U_d
  int *nu = reinterpret_cast<int *>(smem + L.nu);          // [b] |U_d|
  float *C = reinterpret_cast<float *>(smem + L.cost);     // [n_max + 1]
  int *par = reinterpret_cast<int *>(smem + L.par);
  int *dep = reinterpret_cast<int *>(smem + L.dep);
  int *tok = reinterpret_cast<int *>(smem + L.tok);
  float *ah = reinterpret_cast<float *>(smem + L.ah);
  float *sp = reinterpret_cast<float *>(smem + L.sp);
  int *ptok = reinterpret_cast<int *>(smem + L.ptok);     // pending child's token (-1: none)
  int *pu = reinterpret_cast<int *>(smem + L.pu);         // pending child's union index
  uint32_t *mask = reinterpret_cast<uint32_t *>(smem + L.mask);    // [n_max][W]
  uint32_t *taken = reinterpret_cast<uint32_t *>(smem + L.taken);  // [n_max][UW]
  int *etok = reinterpret_cast<int *>(smem + L.etok);      // [E] one position's entries
  int *efirst = reinterpret_cast<int *>(smem + L.efirst);  // [E] first entry with that token
  int *umap = reinterpret_cast<int *>(smem + L.umap);      // [E] union index of a first entry

  griddep_wait();
  griddep_launch_dependents();

  // ---- tables: lse sums and log pi per branch, the cost row
  const double *lse_r = a.lse + (size_t)r * Z * b;
  if (lane < Z) {
    double s = 0.0;
    Lam[lane * (b + 1)] = 0.0;
    for (int d = 1; d <= b; ++d) {
      s += lse_r[(size_t)lane * b + d - 1];
      Lam[lane * (b + 1) + d] = s;
    }
    const double w = a.pi[(size_t)r * Z + lane];
    lpi[lane] = log(w);
    if (!(w >= 0.0) || isinf(w)) atomicOr(&a.status[r], BASTION_STATUS_BAD_WEIGHT);
  }
  const float *cr = a.cost + (a.cost_per_request ? (size_t)r * (n_max + 1) : 0);
  bool bad = false;
  for (int i = lane; i <= n_max; i += 32) {
    const float c = cr[i];
    C[i] = c;
    if (i >= 1) bad |= !(c > 0.f) || isinf(c);
  }
  if (__any_sync(kFull, bad) && lane == 0) atomicOr(&a.status[r], BASTION_STATUS_BAD_COST);

  // ---- the union of the branches' tokens at each position; entry e is
  // (branch e / K, rank e % K)
  const size_t rb = (size_t)r * Z * b * K;
  for (int d = 0; d < b; ++d) {
    for (int e = lane; e < E; e += 32)
      etok[e] = a.topk_tok[rb + ((size_t)(e / K) * b + d) * K + (e % K)];
    __syncwarp();
    for (int e = lane; e < E; e += 32) {
      const int t = etok[e];
      int f = e;
      for (int e2 = 0; e2 < e; ++e2)
        if (etok[e2] == t) {
          f = e2;
          break;
        }
      efirst[e] = f;
    }
    __syncwarp();
    int cnt = 0;
    for (int base = 0; base < E; base += 32) {
      const int e = base + lane;
      const bool first = e < E && efirst[e] == e;
      const uint32_t bal = __ballot_sync(kFull, first);
      if (first) {
        const int u = cnt + __popc(bal & ((1u << lane) - 1u));
        umap[e] = u;
        utok[d * E + u] = etok[e];
      }
      cnt += __popc(bal);
    }
    if (lane == 0) nu[d] = cnt;
    for (int q = lane; q < cnt * Z; q += 32) ulg[(size_t)d * E * Z + q] = -INFINITY;
    __syncwarp();
    for (int e = lane; e < E; e += 32) {
      const int u = umap[efirst[e]];
      ulg[((size_t)d * E + u) * Z + e / K] = a.topk_logit[rb + ((size_t)(e / K) * b + d) * K + (e % K)];
    }
    __syncwarp();
  }

  // log rho of child u (position dq of the union) of node q
  auto child_lr = [&](int q, int dq, int u) -> double {
    double t[8];
    double m = kNegInf;
    for (int z = 0; z < Z; ++z) {
      const double lv = (double)ulg[((size_t)dq * E + u) * Z + z];
      const double lq = Ls[q * Z + z];
      const double ls = (lq == kNegInf || lv == kNegInf) ? kNegInf : lq + lv;
      t[z] = ls == kNegInf ? kNegInf : lpi[z] + (ls - Lam[z * (b + 1) + dq + 1]);
      m = t[z] > m ? t[z] : m;
    }
    if (m == kNegInf) return kNegInf;
    double s = 0.0;
    for (int z = 0; z < Z; ++z) s += exp(t[z] - m);
    return m + log(s);
  };
  // node q's best untaken child -> (plr, ptok, pu); ptok = -1 when none
  auto rescan = [&](int q) {
    const int dq = dep[q];
    double bs = kNegInf;
    int bt = -1, bu = -1;
    if (dq < b) {
      const int n_u = nu[dq];
      for (int u = lane; u < n_u; u += 32) {
        if ((taken[q * UW + (u >> 5)] >> (u & 31)) & 1u) continue;
        const double s = child_lr(q, dq, u);
        const int t = utok[dq * E + u];
        if (bt < 0 || s > bs || (s == bs && t < bt)) {
          bs = s;
          bt = t;
          bu = u;
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const double s2 = __shfl_xor_sync(kFull, bs, o);
      const int t2 = __shfl_xor_sync(kFull, bt, o);
      const int u2 = __shfl_xor_sync(kFull, bu, o);
      const bool take = t2 >= 0 && (bt < 0 || s2 > bs || (s2 == bs && t2 < bt));
      bs = take ? s2 : bs;
      bt = take ? t2 : bt;
      bu = take ? u2 : bu;
    }
    if (lane == 0) {
      plr[q] = bs;
      ptok[q] = bt;
      pu[q] = bu;
    }
    __syncwarp();
  };

  // ---- the root
  const double Lar = (double)a.l_ar[r];
  if (lane == 0) {
    par[0] = -1;
    dep[0] = 0;
    tok[0] = a.root_token[r];
    lr[0] = 0.0;
  }
  if (lane < Z) Ls[lane] = 0.0;
  for (int w = lane; w < W; w += 32) mask[w] = w == 0 ? 1u : 0u;
  for (int q = lane; q < n_max * UW; q += 32) taken[q] = 0u;
  __syncwarp();
  double A = 1.0;
  if (lane == 0) {
    ah[0] = 1.f;
    sp[0] = (float)(A * Lar / (double)C[1]);
  }
  __syncwarp();
  rescan(0);

  int N = 1;
  while (N < n_max) {
    // the best pending candidate over the nodes
    double bs = kNegInf;
    int bd = 0, bt = -1, bn = -1;
    for (int q = lane; q < N; q += 32) {
      const int t = ptok[q];
      if (t < 0) continue;
      const double s = plr[q];
      const int d = dep[q] + 1;
      if (bn < 0 || mix_better(s, d, t, q, bs, bd, bt, bn)) {
        bs = s;
        bd = d;
        bt = t;
        bn = q;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const double s2 = __shfl_xor_sync(kFull, bs, o);
      const int d2 = __shfl_xor_sync(kFull, bd, o);
      const int t2 = __shfl_xor_sync(kFull, bt, o);
      const int n2 = __shfl_xor_sync(kFull, bn, o);
      const bool take = n2 >= 0 && (bn < 0 || mix_better(s2, d2, t2, n2, bs, bd, bt, bn));
      bs = take ? s2 : bs;
      bd = take ? d2 : bd;
      bt = take ? t2 : bt;
      bn = take ? n2 : bn;
    }
    // no candidate, or the best has rho = 0 (a NaN score, from a bad weight,
    // counts as rho = 0 too)
    if (bn < 0 || !(bs > kNegInf)) break;
    const double rho = exp(bs);
    if ((A + rho) * Lar / (double)C[N + 1] < A * Lar / (double)C[N]) break;  // S would decrease
    const int p = bn, i = N, u = pu[p], dp = dep[p];
    N = i + 1;
    A += rho;
    if (lane < Z) {
      const double lv = (double)ulg[((size_t)dp * E + u) * Z + lane];
      const double lq = Ls[p * Z + lane];
      Ls[i * Z + lane] = (lq == kNegInf || lv == kNegInf) ? kNegInf : lq + lv;
    }
    for (int w = lane; w < W; w += 32)
      mask[i * W + w] = mask[p * W + w] | (w == (i >> 5) ? (1u << (i & 31)) : 0u);
    if (lane == 0) {
      par[i] = p;
      dep[i] = bd;
      tok[i] = bt;
      lr[i] = bs;
      ah[i] = (float)A;
      sp[i] = (float)(A * Lar / (double)C[N]);
      taken[p * UW + (u >> 5)] |= 1u << (u & 31);
    }
    __syncwarp();
    rescan(p);
    rescan(i);
  }
  __syncwarp();

  // ---- outputs
  const size_t nb = (size_t)r * n_max;
  const int ctx = a.ctx_len[r];
  if (lane == 0) a.n_nodes[r] = N;
  for (int i = lane; i < N; i += 32) {
    a.parent[nb + i] = par[i];
    a.depth[nb + i] = dep[i];
    a.pos_id[nb + i] = ctx + dep[i];
    a.token[nb + i] = tok[i];
    a.log_rho[nb + i] = (float)lr[i];
    a.a_hat[nb + i] = ah[i];
    a.speedup[nb + i] = sp[i];
  }
  for (int q = lane; q < N * W; q += 32) a.anc_mask[nb * W + q] = mask[q];
}

}  // namespace

size_t mixture_tree_smem_bytes(int Z, int b, int K, int n_max) {
  const int E = Z * K, W = (n_max + 31) / 32, UW = (E + 31) / 32;
  return mix_layout(Z, b, E, n_max, W, UW).bytes;
}

int launch_build_tree_mixture(const float *topk_logit, const int32_t *topk_tok, const double *lse,
                              const double *pi, int B, int Z, int b, int K, int n_max,
                              const int32_t *root_token, const int32_t *ctx_len,
                              const float *cost_ms, int cost_per_request, const float *l_ar,
                              int32_t *n_nodes, int32_t *parent, int32_t *depth, int32_t *pos_id,
                              int32_t *token, float *log_rho, float *a_hat, float *speedup,
                              uint32_t *anc_mask, int32_t *status, cudaStream_t stream) {
  MixArgs a;
  a.topk_logit = topk_logit;
  a.topk_tok = topk_tok;
  a.lse = lse;
  a.pi = pi;
  a.B = B;
  a.Z = Z;
  a.b = b;
  a.K = K;
  a.n_max = n_max;
  a.W = (n_max + 31) / 32;
  a.E = Z * K;
  a.UW = (a.E + 31) / 32;
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
  a.log_rho = log_rho;
  a.a_hat = a_hat;
  a.speedup = speedup;
  a.anc_mask = anc_mask;
  a.status = status;
  const size_t smem = mixture_tree_smem_bytes(Z, b, K, n_max);
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(build_tree_mixture_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return BASTION_ERR_LAUNCH;
  const cudaError_t e = launch_pdl(build_tree_mixture_kernel, dim3(B), dim3(32), smem, stream, a);
  return (e == cudaSuccess && cudaGetLastError() == cudaSuccess) ? BASTION_OK : BASTION_ERR_LAUNCH;
}

}  // namespace bastion
