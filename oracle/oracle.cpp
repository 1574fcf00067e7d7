// CPU oracle for the BASTION draft-tree hot path.  TEST INFRASTRUCTURE ONLY.
//
// A plain, slow, single-threaded fp64 statement of what the hot path computes,
// used by the tests, the smoke check and the bench's CPU-baseline leg to check
// and time the CUDA library.  It shares no code, header, table or helper with
// the CUDA side, and the product path never calls it.
//
// Source of the method: "Bastion: Budget-Aware Speculative Decoding with
// Tree-structured Block Diffusion Drafting" (gist.science/nl/paper/2605.29727,
// Dutch technical summary; the French page gist.science/fr/paper/2605.29727
// carries the same text), section "Methodologie":
//   §1 "Pad-scoren": rho(i) = prod_{k<=d(i)} q_k(x_ik) over the block-diffusion
//      marginals q_k;
//   §2 "Surrogaat-schatting": A_hat(T) = sum_{i in T} rho(i); "Optimale
//      Constructie": repeatedly add the valid node with the highest rho;
//   §3 "Adaptief Stoppen": grow until S(N) = A_hat(T_N) * L_AR / C(N) starts to
//      decrease;
//   "Experimentele Resultaten": verification is greedy (temperature 0).
// Where the pages are silent the readings used are stated at each function.
//
// Parity status: every function here is pinned by tests that do not reuse its
// arithmetic (brute force, closed forms, library routines, invariants), except
// the premise that A_hat predicts real acceptance, which needs trained models
// and is not exercised (parity unpinned for that premise only).

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <vector>

namespace {

const double kInf = std::numeric_limits<double>::infinity();

double load_logit(const void* base, int dtype, int64_t idx) {
  if (dtype == 0) return (double)((const float*)base)[idx];
  if (dtype == 2) return ((const double*)base)[idx];
  uint32_t bits = (uint32_t)((const uint16_t*)base)[idx] << 16;
  float f;
  std::memcpy(&f, &bits, 4);
  return (double)f;
}

double bf16_to_double(uint16_t h) {
  uint32_t bits = (uint32_t)h << 16;
  float f;
  std::memcpy(&f, &bits, 4);
  return (double)f;
}

}  // namespace

extern "C" {

// Status bits written per row / per request by the oracle.
enum { OR_NONFINITE = 1, OR_EMPTY_ROW = 2, OR_BAD_COST = 4 };

// ---------------------------------------------------------------------------
// Step 1: marginals q_k = softmax(l_k) and the K best tokens of each position.
// ("Methodologie" §1: the drafter yields position-wise marginals {q_k}; the
// ranking of candidate tokens per position is the plain order of q_k.)
//
// Reading: q_k at temperature 1; ties in rank are broken by lower token id.
// Outputs per row: the K best logits as given (topk_logit, exact), their
// tokens, log q = l - lse rounded to float (topk_logq), and lse in fp64.
//
// logits: rows x V values (dtype 0 = float32, 1 = bfloat16 bits, 2 = double),
// row stride ld.
int oracle_topk_marginals(const void* logits, int dtype, int rows, int V, int64_t ld, int K,
                          float* topk_logq, float* topk_logit, int32_t* topk_tok,
                          double* lse_f64, int32_t* row_status) {
  if (rows < 0 || V < 1 || K < 1 || K > V || ld < V) return -1;
  std::vector<double> l(V);
  std::vector<int32_t> idx(V);
  for (int r = 0; r < rows; ++r) {
    int st = 0;
    double m = -kInf;
    for (int v = 0; v < V; ++v) {
      l[v] = load_logit(logits, dtype, (int64_t)r * ld + v);
      if (std::isnan(l[v]) || l[v] == kInf) st |= OR_NONFINITE;
      if (l[v] > m) m = l[v];
    }
    if (m == -kInf) st |= OR_EMPTY_ROW;
    // log-sum-exp with the max shifted out
    double s = 0.0;
    for (int v = 0; v < V; ++v) s += std::exp(l[v] - m);
    double lse = m + std::log(s);
    // rank: logit descending, token ascending
    for (int v = 0; v < V; ++v) idx[v] = v;
    std::partial_sort(idx.begin(), idx.begin() + K, idx.end(), [&](int32_t a, int32_t b) {
      if (l[a] != l[b]) return l[a] > l[b];
      return a < b;
    });
    for (int j = 0; j < K; ++j) {
      int32_t v = idx[j];
      topk_tok[(int64_t)r * K + j] = v;
      topk_logq[(int64_t)r * K + j] = (float)(l[v] - lse);
      topk_logit[(int64_t)r * K + j] = (float)l[v];
    }
    lse_f64[r] = lse;
    if (row_status) row_status[r] = st;
  }
  return 0;
}

// ---------------------------------------------------------------------------
// Steps 2-3: best-first prefix-tree expansion under the online controller, and
// the emitted tree arrays.
//
// "Methodologie" §1 (path score rho, prefix tree from position-wise candidates;
// candidates at different positions combine freely), §2 (A_hat = sum rho; add
// the valid node with the highest rho), §3 (stop when S(N) = A_hat*L_AR/C(N)
// starts to decrease).
//
// Readings:
//  * The root (the last committed token) is node 0 at depth 0 with rho = 1 (the
//    empty product) and is counted in N and in A_hat (root_counts = 1).  With
//    root_counts = 0 the root is still emitted as node 0 but N and A_hat count
//    only draft nodes (the alternative reading; S(N) then uses C(#draft)).
//  * The children of a depth-d node are the K ranked tokens of q_{d+1}; depth
//    is at most b.
//  * Candidate order: log rho descending, then depth, rank, token id and parent
//    node index ascending (a total order).
//  * Stop rule: start from T_1 = {root}; for N = 2..n_max take the best
//    candidate c; if S(N) < S(N-1) strictly, stop with T_{N-1}; else add c.
//    Also stop when no candidate is left or the best has log rho = -inf.
//  * log rho of a depth-d node = sum_{k<=d} log q_k(x_k) is evaluated as
//    (sum of the path's logits) - (lse_1 + ... + lse_d): both sums in fp64,
//    accumulated from the root down.  Paths of equal depth then compare on
//    their logit sums alone, which are exact, so equal-depth order and equal-depth
//    ties do not depend on how lse was rounded.
//
// Near ties (several correct results): a pop is flagged when a candidate at a
// different depth than the best is within 1e-6 of it in log rho (there the
// order depends on the lse values' last bits); a stop test is flagged when
// |rho_c C(N-1) - A_hat(N-1) (C(N) - C(N-1))| < 1e-6 A_hat(N-1) |C(N) - C(N-1)|.
// With a guide (another implementation's tree), the oracle follows the guide at
// a flagged step only, and only when the guide's choice is itself within the
// 1e-6 band of the oracle's best; every other step is the oracle's own.
//
// Inputs:  topk_logit/topk_tok [B, b, K]; lse [B, b] (fp64); root_token, ctx_len [B]; cost_ms
// [Bc, n_max+1] with entry N = C(N) (Bc = B if cost_per_request else 1); l_ar [B].
// Outputs: n_nodes [B]; per node [B, n_max]: parent (root -1), depth, pos_id
// (= ctx_len + depth), token, rank (root -1), log_rho, a_hat (A_hat of the
// tree made of nodes 0..n), speedup (S at that size); anc_mask [B, n_max, W]
// (W = ceil(n_max/32); bit j of word j/32: node j is an ancestor of, or is,
// the node); status [B].  Counters: flagged pops, flagged stops, guided steps.
int oracle_build_tree(const float* topk_logit, const int32_t* topk_tok, const double* lse,
                      int B, int b, int K,
                      int n_max, const int32_t* root_token, const int32_t* ctx_len,
                      const float* cost_ms, int cost_per_request, const float* l_ar,
                      int root_counts, const int32_t* guide_n_nodes,
                      const int32_t* guide_parent, const int32_t* guide_rank,
                      int32_t* n_nodes, int32_t* parent, int32_t* depth, int32_t* pos_id,
                      int32_t* token, int32_t* rank, double* log_rho, double* a_hat,
                      double* speedup, uint32_t* anc_mask, int32_t* status,
                      int32_t* n_flag_pop, int32_t* n_flag_stop, int32_t* n_guided) {
  if (B < 0 || b < 1 || K < 1 || n_max < 1) return -1;
  const int W = (n_max + 31) / 32;
  int flag_pop = 0, flag_stop = 0, guided = 0;
  for (int r = 0; r < B; ++r) {
    const float* lg = topk_logit + (int64_t)r * b * K;
    std::vector<double> Lam(b + 1, 0.0);  // Lam[d] = lse_1 + ... + lse_d
    for (int d = 1; d <= b; ++d) Lam[d] = Lam[d - 1] + lse[(int64_t)r * b + d - 1];
    std::vector<double> Lsum(n_max, 0.0);  // per tree node: sum of its path's logits
    const int32_t* tk = topk_tok + (int64_t)r * b * K;
    const float* C = cost_ms + (cost_per_request ? (int64_t)r * (n_max + 1) : 0);
    const double L = (double)l_ar[r];
    int32_t* par = parent + (int64_t)r * n_max;
    int32_t* dep = depth + (int64_t)r * n_max;
    int32_t* pos = pos_id + (int64_t)r * n_max;
    int32_t* tok = token + (int64_t)r * n_max;
    int32_t* rk = rank + (int64_t)r * n_max;
    double* lr = log_rho + (int64_t)r * n_max;
    double* ah = a_hat + (int64_t)r * n_max;
    double* sp = speedup + (int64_t)r * n_max;
    uint32_t* mk = anc_mask + (int64_t)r * n_max * W;
    int st = 0;
    for (int N = 1; N <= n_max; ++N)
      if (!(C[N] > 0.0f) || std::isinf(C[N])) st |= OR_BAD_COST;

    // tree = node 0 (root)
    std::vector<std::vector<char>> taken;  // per node: which ranks are in the tree
    int n = 1;
    par[0] = -1; dep[0] = 0; pos[0] = ctx_len[r]; tok[0] = root_token[r]; rk[0] = -1;
    lr[0] = 0.0;
    for (int w = 0; w < W; ++w) mk[w] = 0;
    mk[0] = 1u;
    taken.assign(n_max, std::vector<char>(K, 0));
    double A = root_counts ? 1.0 : 0.0;        // A_hat of the current tree
    auto counted = [&](int size) { return root_counts ? size : size - 1; };
    auto S_of = [&](double a, int size) { return a * L / (double)C[counted(size)]; };
    ah[0] = A;
    sp[0] = counted(1) >= 1 ? S_of(A, 1) : 0.0;

    while (n < n_max) {
      // explicit candidate list: every (tree node p, rank j) not yet in the tree
      struct Cand { double lr, ls; int d, j, t, p; };
      auto better = [](const Cand& x, const Cand& y) {
        if (x.lr != y.lr) return x.lr > y.lr;
        if (x.d != y.d) return x.d < y.d;
        if (x.j != y.j) return x.j < y.j;
        if (x.t != y.t) return x.t < y.t;
        return x.p < y.p;
      };
      std::vector<Cand> cands;
      for (int p = 0; p < n; ++p) {
        if (dep[p] >= b) continue;
        int d = dep[p] + 1;
        for (int j = 0; j < K; ++j) {
          if (taken[p][j]) continue;
          double ls = Lsum[p] + (double)lg[(int64_t)(d - 1) * K + j];
          cands.push_back({ls - Lam[d], ls, d, j, tk[(int64_t)(d - 1) * K + j], p});
        }
      }
      if (cands.empty()) break;
      int best = 0;
      for (int c = 1; c < (int)cands.size(); ++c)
        if (better(cands[c], cands[best])) best = c;
      // near-tie check on the pop (only rivals at another depth can be ambiguous)
      bool pop_flag = false;
      for (int c = 0; c < (int)cands.size(); ++c)
        if (c != best && cands[c].d != cands[best].d && cands[best].lr - cands[c].lr < 1e-6)
          pop_flag = true;
      if (pop_flag) ++flag_pop;
      int choice = best;
      if (pop_flag && guide_parent && guide_n_nodes && n < guide_n_nodes[r]) {
        int gp = guide_parent[(int64_t)r * n_max + n], gj = guide_rank[(int64_t)r * n_max + n];
        for (int c = 0; c < (int)cands.size(); ++c)
          if (cands[c].p == gp && cands[c].j == gj &&
              cands[best].lr - cands[c].lr < 1e-6) {
            if (c != best) ++guided;
            choice = c;
            break;
          }
      }
      const Cand& c = cands[choice];
      if (c.lr == -kInf) break;
      // controller: S(N) against S(N-1), N = n + 1
      double rho = std::exp(c.lr);
      int size_new = n + 1;
      double S_prev = S_of(A, n);
      double S_new = S_of(A + rho, size_new);
      bool stop = counted(n) >= 1 ? (S_new < S_prev) : false;
      double dC = (double)C[counted(size_new)] - (double)(counted(n) >= 0 ? C[counted(n)] : 0.0f);
      if (counted(n) >= 1 && dC != 0.0) {
        double margin = rho * (double)C[counted(n)] - A * dC;
        if (std::fabs(margin) < 1e-6 * A * std::fabs(dC)) {
          ++flag_stop;
          if (guide_n_nodes) {
            bool gstop = guide_n_nodes[r] == n;
            if (gstop != stop) ++guided;
            stop = gstop;
          }
        }
      }
      if (stop) break;
      // add the node
      int i = n++;
      taken[c.p][c.j] = 1;
      A += rho;
      par[i] = c.p; dep[i] = c.d; pos[i] = ctx_len[r] + c.d; tok[i] = c.t; rk[i] = c.j;
      lr[i] = c.lr; Lsum[i] = c.ls; ah[i] = A; sp[i] = S_of(A, n);
      for (int w = 0; w < W; ++w) mk[(int64_t)i * W + w] = mk[(int64_t)c.p * W + w];
      mk[(int64_t)i * W + i / 32] |= 1u << (i % 32);
    }
    n_nodes[r] = n;
    if (status) status[r] = st;
  }
  if (n_flag_pop) *n_flag_pop = flag_pop;
  if (n_flag_stop) *n_flag_stop = flag_stop;
  if (n_guided) *n_guided = guided;
  return 0;
}

// ---------------------------------------------------------------------------
// Step 4: greedy (temperature 0) verification ("Experimentele Resultaten":
// evaluation with greedy decoding).  The target's greedy token at each tree node
// is the argmax of that node's target logits (ties: lowest token id).  Starting
// at the root, the draft token equal to the current node's greedy token is
// accepted if it is a child of the current node; the first node with no such
// child ends the walk, and its greedy token is the bonus token.
//
// Outputs: argmax [B, n_max] (rows past n_nodes untouched); accept_len [B];
// accept_nodes [B, b+1] (root, then the accepted nodes, then -1);
// out_tokens [B, b+1] (accepted tokens, then the bonus, then -1).
int oracle_verify_greedy(const void* target, int dtype, int B, int n_max, int V, int64_t ld,
                         int b, const int32_t* n_nodes, const int32_t* parent,
                         const int32_t* token, int32_t* argmax, int32_t* accept_len,
                         int32_t* accept_nodes, int32_t* out_tokens, int32_t* status) {
  if (B < 0 || n_max < 1 || V < 1 || ld < V || b < 1) return -1;
  for (int r = 0; r < B; ++r) {
    int st = 0;
    int nn = n_nodes[r];
    for (int i = 0; i < nn; ++i) {
      int64_t row = ((int64_t)r * n_max + i) * ld;
      int best = 0;
      double bv = load_logit(target, dtype, row);
      for (int v = 0; v < V; ++v) {
        double x = load_logit(target, dtype, row + v);
        if (std::isnan(x) || x == kInf) st |= OR_NONFINITE;
        if (x > bv) { bv = x; best = v; }
      }
      argmax[(int64_t)r * n_max + i] = best;
    }
    int32_t* an = accept_nodes + (int64_t)r * (b + 1);
    int32_t* ot = out_tokens + (int64_t)r * (b + 1);
    for (int k = 0; k <= b; ++k) { an[k] = -1; ot[k] = -1; }
    int cur = 0, len = 0;
    an[0] = 0;
    while (true) {
      int t = argmax[(int64_t)r * n_max + cur];
      int next = -1;
      for (int c = 1; c < nn; ++c)
        if (parent[(int64_t)r * n_max + c] == cur && token[(int64_t)r * n_max + c] == t) {
          next = c;
          break;
        }
      if (next < 0 || len >= b) break;
      ot[len] = t;
      ++len;
      an[len] = next;
      cur = next;
    }
    ot[len] = argmax[(int64_t)r * n_max + cur];
    accept_len[r] = len;
    if (status) status[r] = st;
  }
  return 0;
}

// ---------------------------------------------------------------------------
// Stochastic verification at temperature T > 0.  The pages evaluate greedy
// decoding only ("Experimentele Resultaten"); for sampled decoding of a tree of
// deterministic candidates the plainest lossless reading is taken: at every
// node i the target's token y_i is a draw from softmax(l_i / T), by inverse
// transform with the caller's uniform u[r][i] in [0, 1):
//   y_i = the smallest v whose cumulative weight C_v = sum_{w <= v} w_w, with
//         w_w = exp((l_w - M) / T) and M the row's largest finite logit,
//         exceeds u * C_{V-1};
// the walk is the greedy walk with y in place of the argmax (accept the child
// of the current node whose token is y while one exists, at most b), and the
// bonus is y at the last accepted node.  Each emitted token is then a draw
// from the target's conditional distribution at its prefix.
//
// margin[r][i] = min(u S - C_{y-1}, C_y - u S) / S with S = C_{V-1}: how close
// the draw lies to a neighbouring token's interval (the tests use it where
// floating point may decide).  A row without a finite logit has S = 0: y = 0,
// margin 0 and the OR_EMPTY_ROW bit; NaN or +inf set OR_NONFINITE.
int oracle_verify_sample(const void* target, int dtype, int B, int n_max, int V, int64_t ld,
                         int b, double T, const double* u, const int32_t* n_nodes,
                         const int32_t* parent, const int32_t* token, int32_t* sampled,
                         double* margin, int32_t* accept_len, int32_t* accept_nodes,
                         int32_t* out_tokens, int32_t* status) {
  if (B < 0 || n_max < 1 || V < 1 || ld < V || b < 1 || !(T > 0.0)) return -1;
  std::vector<double> w((size_t)V);
  for (int r = 0; r < B; ++r) {
    int st = 0;
    const int nn = n_nodes[r];
    for (int i = 0; i < nn; ++i) {
      const int64_t row = ((int64_t)r * n_max + i) * ld;
      const int64_t o = (int64_t)r * n_max + i;
      double M = -kInf;
      for (int v = 0; v < V; ++v) {
        const double x = load_logit(target, dtype, row + v);
        if (std::isnan(x) || x == kInf) st |= OR_NONFINITE;
        else if (x > M) M = x;
      }
      double S = 0.0;
      for (int v = 0; v < V; ++v) {
        const double x = load_logit(target, dtype, row + v);
        w[(size_t)v] = (M == -kInf || std::isnan(x) || x == -kInf) ? 0.0 : std::exp((x - M) / T);
        S += w[(size_t)v];
      }
      if (!(S > 0.0)) {
        st |= OR_EMPTY_ROW;
        sampled[o] = 0;
        margin[o] = 0.0;
        continue;
      }
      const double t = u[o] * S;
      double C = 0.0;
      int y = V - 1;
      double lo = 0.0, hi = S;
      for (int v = 0; v < V; ++v) {
        const double Cn = C + w[(size_t)v];
        if (Cn > t) {
          y = v;
          lo = C;
          hi = Cn;
          break;
        }
        C = Cn;
      }
      sampled[o] = y;
      margin[o] = std::min(t - lo, hi - t) / S;
    }
    int32_t* an = accept_nodes + (int64_t)r * (b + 1);
    int32_t* ot = out_tokens + (int64_t)r * (b + 1);
    for (int k = 0; k <= b; ++k) { an[k] = -1; ot[k] = -1; }
    int cur = 0, len = 0;
    an[0] = 0;
    if (nn >= 1) {
      while (true) {
        const int y = sampled[(int64_t)r * n_max + cur];
        int next = -1;
        for (int c = 1; c < nn; ++c)
          if (parent[(int64_t)r * n_max + c] == cur && token[(int64_t)r * n_max + c] == y) {
            next = c;
            break;
          }
        if (next < 0 || len >= b) break;
        ot[len] = y;
        ++len;
        an[len] = next;
        cur = next;
      }
      ot[len] = sampled[(int64_t)r * n_max + cur];
    }
    accept_len[r] = len;
    if (status) status[r] = st;
  }
  return 0;
}

// ---------------------------------------------------------------------------
// Calibration of the verification cost model ("Methodologie" §3,
// "Latentiemodellering": T_verify(N) comes from a hardware-aware roofline model
// of memory bandwidth and compute, calibrated with observed runtimes to correct
// for kernel fusion and scheduling overhead).
//
// Reading: the roofline of a target forward over N tree tokens is
//   roof(N) = max((bytes0 + bytes1 N) / bw, (flops0 + flops1 N) / peak)   [ms]
// and the calibration is the least-squares line T_verify = alpha roof + beta
// through the observed samples (N_i, t_i ms).  When the samples' roofline
// values have no spread, alpha = 1 and beta = mean(t - roof).  The table the
// tree controller reads is C(N) = t_draft + alpha roof(N) + beta for
// N = 0 .. n_max.
//
// out_params = {alpha, beta}.  Returns -1 on bad arguments.
int oracle_calibrate_cost(const double* sample_n, const double* sample_ms, int n_samples,
                          double bytes0, double bytes1, double flops0, double flops1, double bw,
                          double peak, double t_draft, int n_max, double* cost_out,
                          double* out_params) {
  if (n_samples < 1 || n_max < 1 || !(bw > 0.0) || !(peak > 0.0)) return -1;
  auto roof = [&](double N) { return std::max((bytes0 + bytes1 * N) / bw, (flops0 + flops1 * N) / peak); };
  double sr = 0.0, st = 0.0;
  for (int k = 0; k < n_samples; ++k) {
    sr += roof(sample_n[k]);
    st += sample_ms[k];
  }
  const double mr = sr / n_samples, mt = st / n_samples;
  double srr = 0.0, srt = 0.0;
  for (int k = 0; k < n_samples; ++k) {
    const double dr = roof(sample_n[k]) - mr;
    srr += dr * dr;
    srt += dr * (sample_ms[k] - mt);
  }
  double alpha = 1.0, beta = mt - mr;
  if (srr > 1e-12 * std::max(1.0, mr * mr) * n_samples) {
    alpha = srt / srr;
    beta = mt - alpha * mr;
  }
  for (int N = 0; N <= n_max; ++N) cost_out[N] = t_draft + alpha * roof((double)N) + beta;
  out_params[0] = alpha;
  out_params[1] = beta;
  return 0;
}

// ---------------------------------------------------------------------------
// Tree-masked GQA attention of the tree's query tokens against the KV cache
// (the target verifies the whole tree in one parallel forward: "Probleemstelling"
// and "Methodologie" §2 of the pages; the mask is what makes that forward
// equal to one sequential pass per root path).
//
// Reading: query i of request r sees every committed context slot j < ctx_len[r]
// and the tree slot ctx_len[r] + t (t < n_nodes[r]) iff node t is an ancestor of
// node i or node i itself (bit t of anc_mask[r][i]); head h reads KV head
// h / (Hq / Hkv); scores are scale * q.k; softmax and the weighted sum in fp64.
//
// q: bf16 bits [B, n_max, Hq, D]; k, v: bf16 bits [B, L_cap, Hkv, D].
// sel: optional list of n_sel (r, i, h) triples (int32 x3); when null every
// (r, i < n_nodes[r], h) is computed in that order.  out: fp64 [n_out, D].
// Returns the number of rows written, or -1 on bad arguments.
int64_t oracle_tree_attention(const uint16_t* q, const uint16_t* k, const uint16_t* v, int B,
                              int n_max, int Hq, int Hkv, int D, int64_t L_cap,
                              const int32_t* ctx_len, const int32_t* n_nodes,
                              const uint32_t* anc_mask, double scale, const int32_t* sel,
                              int64_t n_sel, double* out) {
  if (B < 0 || n_max < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv || D < 1) return -1;
  const int W = (n_max + 31) / 32;
  const int G = Hq / Hkv;
  std::vector<double> sc;
  auto one = [&](int r, int i, int h, double* o) {
    int ctx = ctx_len[r], nn = n_nodes[r];
    int hk = h / G;
    const uint16_t* qv = q + (((int64_t)r * n_max + i) * Hq + h) * D;
    int64_t nk = (int64_t)ctx + nn;
    sc.assign(nk, -kInf);
    double m = -kInf;
    for (int64_t j = 0; j < nk; ++j) {
      bool vis = j < ctx;
      if (!vis) {
        int t = (int)(j - ctx);
        vis = (anc_mask[((int64_t)r * n_max + i) * W + t / 32] >> (t % 32)) & 1u;
      }
      if (!vis) continue;
      const uint16_t* kv = k + (((int64_t)r * L_cap + j) * Hkv + hk) * D;
      double dot = 0.0;
      for (int d = 0; d < D; ++d) dot += bf16_to_double(qv[d]) * bf16_to_double(kv[d]);
      sc[j] = scale * dot;
      if (sc[j] > m) m = sc[j];
    }
    double den = 0.0;
    for (int64_t j = 0; j < nk; ++j)
      if (sc[j] != -kInf) den += std::exp(sc[j] - m);
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    for (int64_t j = 0; j < nk; ++j) {
      if (sc[j] == -kInf) continue;
      double p = std::exp(sc[j] - m) / den;
      const uint16_t* vv = v + (((int64_t)r * L_cap + j) * Hkv + hk) * D;
      for (int d = 0; d < D; ++d) o[d] += p * bf16_to_double(vv[d]);
    }
  };
  int64_t cnt = 0;
  if (sel) {
    for (int64_t s = 0; s < n_sel; ++s) {
      one(sel[3 * s], sel[3 * s + 1], sel[3 * s + 2], out + cnt * D);
      ++cnt;
    }
  } else {
    for (int r = 0; r < B; ++r)
      for (int i = 0; i < n_nodes[r]; ++i)
        for (int h = 0; h < Hq; ++h) {
          one(r, i, h, out + cnt * D);
          ++cnt;
        }
  }
  return cnt;
}

// ---------------------------------------------------------------------------
// Latent-mixture trees.  DBlast (the third page on this subject, "Methodologie"
// 1, "Afhankelijke Blok-sampling via Latente Mix") replaces the factorised
// block proposal by a mixture over a latent branch z:
//   q_dep(x_1..b | y) = sum_z q(z|y) prod_i q_i(x_i | y, z).
// The tree of Bastion's §1-§3 is grown on the path score this induces: the
// mixture probability of a prefix,
//   rho(x_1..d) = sum_z pi_z prod_{k<=d} q_k^z(x_k),   pi_z = q(z|y),
// which is non-increasing along a path (every term is), so best-first on it
// still yields, for every N, the prefix-closed tree of N nodes with the largest
// sum of rho (the nodes with the N largest scores).
//
// Readings:
//  * Each branch keeps its K ranked tokens per position (step 1 applied per
//    branch); a token outside branch z's list at position k has q_k^z = 0.
//  * The children of a depth-d node are the union over z of the branches'
//    tokens at position d+1; depth is at most b.
//  * Per branch, log of the path product = (sum of the path's logits in that
//    branch) - (that branch's lse_1 + ... + lse_d), both sums in fp64 (-inf when
//    a token is missing from the branch); log rho = log sum_z exp(log pi_z +
//    that), taken with the largest term factored out.
//  * Candidate order: log rho descending, then depth, token id and parent node
//    index ascending.  The root is node 0 with rho = 1 (sum_z pi_z, the caller
//    passes pi summing to 1) and is counted in N and A_hat; the stop rule is
//    step 2's.
//
// Near ties (several correct results).  Unlike the single-proposal tree, two
// candidates of equal depth are not compared on exact logit sums: log rho is a
// log-sum-exp over the branches, and an implementation that forms it in
// single precision is off by a few 1e-6.  So the band is 1e-5 here: a pop is
// flagged when another candidate is within 1e-5 of the best in log rho, unless
// it has the same parent and the same logit in every branch (then log rho is
// the same function of the same numbers on any implementation, and the token
// order decides); a stop test is flagged when
// |rho_c C(N) - A_hat (C(N+1) - C(N))| < 1e-5 A_hat |C(N+1) - C(N)|.
// With a guide (another implementation's tree: n_nodes, and parent and token
// per node), the oracle follows the guide at a flagged step only, and only
// when the guide's choice is itself within the band of the oracle's best.
//
// Inputs: topk_logit/topk_tok [B, Z, b, K]; lse [B, Z, b]; pi [B, Z];
// root_token, ctx_len [B]; cost_ms [Bc, n_max+1]; l_ar [B]; the guide (may be
// null).  Outputs as step 2 without rank: n_nodes; parent, depth, pos_id,
// token, log_rho, a_hat, speedup [B, n_max]; anc_mask [B, n_max, W]; status
// [B]; counters (may be null): flagged pops, flagged stops, guided steps.
int oracle_build_tree_mixture(const float* topk_logit, const int32_t* topk_tok, const double* lse,
                              const double* pi, int B, int Z, int b, int K, int n_max,
                              const int32_t* root_token, const int32_t* ctx_len,
                              const float* cost_ms, int cost_per_request, const float* l_ar,
                              const int32_t* guide_n_nodes, const int32_t* guide_parent,
                              const int32_t* guide_token,
                              int32_t* n_nodes, int32_t* parent, int32_t* depth, int32_t* pos_id,
                              int32_t* token, double* log_rho, double* a_hat, double* speedup,
                              uint32_t* anc_mask, int32_t* status, int32_t* n_flag_pop,
                              int32_t* n_flag_stop, int32_t* n_guided) {
  if (B < 0 || Z < 1 || b < 1 || K < 1 || n_max < 1) return -1;
  const int W = (n_max + 31) / 32;
  const double kBand = 1e-5;
  int flag_pop = 0, flag_stop = 0, guided = 0;
  for (int r = 0; r < B; ++r) {
    // branch z, position k (0-based), rank j
    auto lg = [&](int z, int k, int j) {
      return (double)topk_logit[(((int64_t)r * Z + z) * b + k) * K + j];
    };
    auto tk = [&](int z, int k, int j) { return topk_tok[(((int64_t)r * Z + z) * b + k) * K + j]; };
    std::vector<std::vector<double>> Lam(Z, std::vector<double>(b + 1, 0.0));
    for (int z = 0; z < Z; ++z)
      for (int d = 1; d <= b; ++d) Lam[z][d] = Lam[z][d - 1] + lse[((int64_t)r * Z + z) * b + d - 1];
    std::vector<double> lpi(Z);
    for (int z = 0; z < Z; ++z) lpi[z] = std::log(pi[(int64_t)r * Z + z]);
    // per node and branch: sum of the path's logits in that branch (-inf if absent)
    std::vector<std::vector<double>> Ls(n_max, std::vector<double>(Z, 0.0));
    auto log_rho_of = [&](const std::vector<double>& ls, int d) {
      double m = -kInf;
      std::vector<double> t(Z);
      for (int z = 0; z < Z; ++z) {
        t[z] = ls[z] == -kInf ? -kInf : lpi[z] + (ls[z] - Lam[z][d]);
        if (t[z] > m) m = t[z];
      }
      if (m == -kInf) return -kInf;
      double s = 0.0;
      for (int z = 0; z < Z; ++z) s += std::exp(t[z] - m);
      return m + std::log(s);
    };
    const float* C = cost_ms + (cost_per_request ? (int64_t)r * (n_max + 1) : 0);
    const double L = (double)l_ar[r];
    int32_t* par = parent + (int64_t)r * n_max;
    int32_t* dep = depth + (int64_t)r * n_max;
    int32_t* pos = pos_id + (int64_t)r * n_max;
    int32_t* tok = token + (int64_t)r * n_max;
    double* lr = log_rho + (int64_t)r * n_max;
    double* ah = a_hat + (int64_t)r * n_max;
    double* sp = speedup + (int64_t)r * n_max;
    uint32_t* mk = anc_mask + (int64_t)r * n_max * W;
    int st = 0;
    for (int N = 1; N <= n_max; ++N)
      if (!(C[N] > 0.0f) || std::isinf(C[N])) st |= OR_BAD_COST;
    int n = 1;
    par[0] = -1; dep[0] = 0; pos[0] = ctx_len[r]; tok[0] = root_token[r]; lr[0] = 0.0;
    for (int w = 0; w < W; ++w) mk[w] = 0;
    mk[0] = 1u;
    std::vector<std::vector<int32_t>> kids(n_max);  // tokens already added under each node
    double A = 1.0;
    auto S_of = [&](double a, int size) { return a * L / (double)C[size]; };
    ah[0] = A;
    sp[0] = S_of(A, 1);
    while (n < n_max) {
      struct Cand { double lr; std::vector<double> ls; int d, t, p; };
      auto better = [](const Cand& x, const Cand& y) {
        if (x.lr != y.lr) return x.lr > y.lr;
        if (x.d != y.d) return x.d < y.d;
        if (x.t != y.t) return x.t < y.t;
        return x.p < y.p;
      };
      std::vector<Cand> cands;
      for (int p = 0; p < n; ++p) {
        if (dep[p] >= b) continue;
        const int d = dep[p] + 1;
        std::vector<int32_t> seen;
        for (int z = 0; z < Z; ++z)
          for (int j = 0; j < K; ++j) {
            const int32_t t = tk(z, d - 1, j);
            if (std::find(seen.begin(), seen.end(), t) != seen.end()) continue;
            seen.push_back(t);
            if (std::find(kids[p].begin(), kids[p].end(), t) != kids[p].end()) continue;
            std::vector<double> ls(Z);
            for (int y = 0; y < Z; ++y) {
              double lv = -kInf;
              for (int i = 0; i < K; ++i)
                if (tk(y, d - 1, i) == t) { lv = lg(y, d - 1, i); break; }
              ls[y] = (Ls[p][y] == -kInf || lv == -kInf) ? -kInf : Ls[p][y] + lv;
            }
            cands.push_back({log_rho_of(ls, d), ls, d, t, p});
          }
      }
      if (cands.empty()) break;
      int best = 0;
      for (int c = 1; c < (int)cands.size(); ++c)
        if (better(cands[c], cands[best])) best = c;
      bool pop_flag = false;
      for (int c = 0; c < (int)cands.size(); ++c)
        if (c != best && cands[best].lr - cands[c].lr < kBand &&
            !(cands[c].p == cands[best].p && cands[c].ls == cands[best].ls))
          pop_flag = true;
      if (pop_flag) ++flag_pop;
      int choice = best;
      if (pop_flag && guide_parent && guide_n_nodes && n < guide_n_nodes[r]) {
        const int gp = guide_parent[(int64_t)r * n_max + n];
        const int gt = guide_token[(int64_t)r * n_max + n];
        for (int c = 0; c < (int)cands.size(); ++c)
          if (cands[c].p == gp && cands[c].t == gt && cands[best].lr - cands[c].lr < kBand) {
            if (c != best) ++guided;
            choice = c;
            break;
          }
      }
      const Cand& c = cands[choice];
      if (c.lr == -kInf) break;
      const double rho = std::exp(c.lr);
      bool stop = S_of(A + rho, n + 1) < S_of(A, n);  // S would decrease: keep T_n
      const double dC = (double)C[n + 1] - (double)C[n];
      if (dC != 0.0 && std::fabs(rho * (double)C[n] - A * dC) < kBand * A * std::fabs(dC)) {
        ++flag_stop;
        if (guide_n_nodes) {
          const bool gstop = guide_n_nodes[r] == n;
          if (gstop != stop) ++guided;
          stop = gstop;
        }
      }
      if (stop) break;
      const int i = n++;
      kids[c.p].push_back(c.t);
      A += rho;
      par[i] = c.p; dep[i] = c.d; pos[i] = ctx_len[r] + c.d; tok[i] = c.t;
      lr[i] = c.lr; Ls[i] = c.ls; ah[i] = A; sp[i] = S_of(A, n);
      for (int w = 0; w < W; ++w) mk[(int64_t)i * W + w] = mk[(int64_t)c.p * W + w];
      mk[(int64_t)i * W + i / 32] |= 1u << (i % 32);
    }
    n_nodes[r] = n;
    if (status) status[r] = st;
  }
  if (n_flag_pop) *n_flag_pop = flag_pop;
  if (n_flag_stop) *n_flag_stop = flag_stop;
  if (n_guided) *n_guided = guided;
  return 0;
}

// ---------------------------------------------------------------------------
// Fused drafter LM-head + top-K.  The drafter's final hidden state h_k of block
// position k times its output embedding W gives that position's logits,
// l_k[v] = W[v] . h_k ("Methodologie" §1: one drafter forward pass yields the
// position-wise marginals q_k = softmax(l_k)); the outputs are those of step 1
// applied to l_k, without the logits ever being an input.
//
// hidden: rows x H, weight: V x H (dtype 0 = float32, 1 = bfloat16 bits).  The
// logits are formed in double: each product of two bf16 or fp32 values is
// exact, and the sum runs over i = 0 .. H-1 in order.  logits_out (optional)
// receives them, rows x V.
int oracle_lm_head_topk(const void* hidden, const void* weight, int dtype, int rows, int H, int V,
                        int K, float* topk_logq, float* topk_logit, int32_t* topk_tok,
                        double* lse_f64, double* logits_out, int32_t* row_status) {
  if (rows < 0 || H < 1 || V < 1 || K < 1 || K > V || (dtype != 0 && dtype != 1)) return -1;
  std::vector<double> h(H), w((size_t)V * H), l(V);
  for (int64_t e = 0; e < (int64_t)V * H; ++e) w[e] = load_logit(weight, dtype, e);
  for (int r = 0; r < rows; ++r) {
    for (int i = 0; i < H; ++i) h[i] = load_logit(hidden, dtype, (int64_t)r * H + i);
    for (int v = 0; v < V; ++v) {
      double s = 0.0;
      for (int i = 0; i < H; ++i) s += w[(size_t)v * H + i] * h[i];
      l[v] = s;
    }
    if (logits_out) std::copy(l.begin(), l.end(), logits_out + (int64_t)r * V);
    const int rc = oracle_topk_marginals(l.data(), 2, 1, V, V, K, topk_logq + (int64_t)r * K,
                                         topk_logit + (int64_t)r * K, topk_tok + (int64_t)r * K,
                                         lse_f64 + r, row_status ? row_status + r : nullptr);
    if (rc != 0) return rc;
  }
  return 0;
}

}  // extern "C"
