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
// a depth-d node are the union U over z of the branches' tokens at position
// d+1.
//
// Arithmetic (no fp64 after the per-request set-up):
//  * Per node n and branch z, P_z(n) = log pi_z + sum over the path of
//    (logit - lse) in branch z, a 64-bit fixed-point integer (2^-40 units) as
//    in the single-proposal tree; -inf where the path leaves branch z's lists.
//  * Position tables: E = exp(logit - max logit of its row) in fp32 for every
//    branch-rank entry, stored per union token and branch.
//  * Node weights: with X_z = P_z(n) + (max logit - lse) of branch z at the
//    children's position and S_n = max_z X_z, w_z(n) = exp(X_z - S_n) in fp32,
//    so the best child of n has sum_z w_z E >= 1.  A child u of n then has
//    rho = exp(S_n) sum_z w_z(n) E_z(u): Z fused multiply-adds in branch order,
//    no transcendental.  Both exponentials reduce their argument in fixed
//    point (x = k ln 2 + f) before one expf, so each is within 2.2 2^-23
//    (relative).
//  * The child's score is S_n + log of that sum, with the log split into
//    exponent * ln 2 (fixed point) and logf of a mantissa in [2^-1/2, 2^1/2):
//    within (5 + Z/2) 2^-23 of the exact log rho (two exponentials, Z
//    roundings of the sum, the log), about 8e-7 for Z = 4 and 2.5e-6 for
//    Z = 32, inside the 1e-5 band of the mixture oracle's near-tie flags.
//  * When a node's best remaining child falls below 2^-100 (its sum loses
//    precision to fp32 underflow), that node's scan is redone in the log
//    domain: the largest branch term of each child in fixed point first, then
//    the sums rescaled by it.
//
// Work layout: one CTA per request.  Its 256 threads stage the tables: the
// request's lists with several loads in flight per thread, the union of each
// position's tokens by hashing into shared memory and a warp-ballot
// compaction, then E per (union token, branch).  Node n's pending candidate,
// its best untaken child, is kept in lane n % 32, register slot n / 32, as a
// 96-bit key (order-preserving image of the score, then a tie word from depth
// and node) with its union index and token, and found by three redux.sync per
// pop.  A pop runs the stop test rho C(N) < A_hat (C(N+1) - C(N)) in fp32 with
// A_hat summed with Kahan compensation, adds the node (lane z forms its P_z
// from the branch's rank of the token and the node's weights from P_z), and
// rescans two child lists: the parent's (its next-best child) and the new
// node's (its best child).
//
// Two forms of the child tables, the same arithmetic in the same order:
//  * dense (Z <= 8, when the tables fit in shared memory): per union token,
//    its E and rank in every branch (padded to ZP = 1, 2, 4 or 8 branches).
//    Four warps run the pops, one per SM sub-partition: each holds the same
//    pending keys and takes the same decisions, and each scans every fourth
//    block of 32 union tokens (one vector load and ZP FMAs per token, the
//    argmax folded in) and owns the taken-bits of those blocks; their four
//    partial argmaxes meet through shared memory at one named barrier per
//    pop (double-buffered, so a warp is at most one pop ahead).  A pop on
//    one warp was bound by instruction issue on a single sub-partition.
//  * sparse (otherwise): E and union index per branch-rank entry; warp 0 runs
//    the pops alone, a scan accumulating per-token sums in shared memory one
//    branch at a time (a branch lists a token at most once, so no two lanes
//    of a pass collide), then taking the argmax.
// Every loop is bounded by the tree budget or a table size; the named barrier
// is reached the same number of times by all four warps (they take identical
// decisions from identical data), and there are no other waits.
#include <climits>
#include <cmath>

#include "common.cuh"
#include "tree_build.cuh"

namespace bastion {

namespace {

using tb::kInfCut;
using tb::kNegFix;

constexpr int kMixThreads = 256;
constexpr int kPopWarps = 4;  // dense form: the warps that run the pops
constexpr int kRootSort = 512;  // dense form: the root's children are sorted once when at most this many
constexpr int64_t kBoundSlack = 1ll << 20;  // 2^-20 in the bounds of lazy entries
constexpr int kEmptySlot = INT_MIN;
constexpr int64_t kLn2Fix = 762123384786ll;  // ln 2 in 2^-40 units, rounded
constexpr int64_t kExpCut = -(104ll << 40);  // exp of less is 0 in fp32
constexpr int64_t kVeryNeg = kNegFix * 2;    // below every finite score
constexpr float kTiny = 7.888609052210118e-31f;  // 2^-100

struct MixArgs {
  const float *topk_logit;  // [B, Z, b, K]
  const int32_t *topk_tok;  // [B, Z, b, K]
  const double *lse;        // [B, Z, b]
  const double *pi;         // [B, Z]
  int B, Z, b, K, n_max;
  const int32_t *root_token, *ctx_len;
  const float *cost;
  int cost_per_request;
  const float *l_ar;
  int32_t *n_nodes, *parent, *depth, *pos_id, *token;
  float *log_rho, *a_hat, *speedup;
  uint32_t *anc_mask;
  int32_t *status;
  unsigned char *ws;  // the requests' tables, ws_stride bytes each
  size_t ws_stride;
};

// One request's tables (region 1), built by the staging kernel in the
// workspace and copied as they are into the pop kernel's shared memory, then
// the pop kernel's own arrays (region 2).  Entry e = (d Z + z) K + j is branch
// z's rank-j token at block position d + 1; union token u of position d + 1
// is slot d ZK + u.  ZP = 0: the sparse form.
struct MixLayout {
  size_t flse, fmax, mq, lq, utok, nu, ue;  // region 1, both forms
  size_t dE, dR;                            // region 1, dense form
  size_t ee;                                // region 1, sparse form
  size_t r1;                                // region 1 bytes
  size_t cost, pn, sn, lrn, acc, wz, an, taken, mask, par, dep, tok, pu, pt, part;  // region 2
  size_t rv, rt, ru, rk, lgn;               // region 2, dense form: the root's sorted children
  int NR;                                   // their capacity (a power of two, 0: none)
  size_t bytes;                             // the pop kernel's shared memory
  int H;                                    // hash slots per position (staging)
};

__host__ __device__ inline MixLayout mix_layout(int Z, int b, int K, int n_max, int ZP) {
  MixLayout l;
  const size_t ZK = (size_t)Z * K, E = (size_t)b * ZK;
  const size_t W = (n_max + 31) / 32, UW = (ZK + 31) / 32, n = (size_t)n_max;
  int H = 64;
  while ((size_t)H < 2 * ZK) H <<= 1;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o += (bytes + 15) & ~(size_t)15;
    return at;
  };
  l.flse = take((size_t)b * Z * 8);
  l.fmax = take((size_t)b * Z * 8);
  l.mq = take((size_t)b * Z * 8);
  l.lq = take(E * 8);
  l.utok = take(E * 4);
  l.nu = take((size_t)b * 4);
  l.ue = take(E * 2);
  l.dE = l.dR = l.ee = 0;
  if (ZP > 0) {
    l.dE = take(E * ZP * 4);
    l.dR = take(E * ZP * 2);
  } else {
    l.ee = take(E * 4);
  }
  l.r1 = o;
  const size_t copies = ZP > 0 ? kPopWarps : 1;  // per-warp copies of P, S, w and the pending child
  l.cost = take((n + 1) * 4);
  l.pn = take(copies * n * Z * 8);
  l.sn = take(copies * n * 8);
  l.lrn = take(n * 8);
  l.acc = ZP > 0 ? 0 : take(2 * ZK * 4);  // also ZK int64 in the log-domain rescan
  l.wz = take(copies * n * Z * 4);
  l.an = take(n * 4);
  l.taken = take(n * UW * 4);
  l.mask = take(n * W * 4);
  l.par = take(n * 4);
  l.dep = take(n * 4);
  l.tok = take(n * 4);
  l.pu = take(copies * n * 4);
  l.pt = take(copies * n * 4);
  l.part = ZP > 0 ? take(2 * 2 * kPopWarps * 16) : 0;
  int NR = 0;
  if (ZP > 0) {
    NR = 32;
    while ((size_t)NR < ZK && NR < kRootSort) NR <<= 1;
  }
  l.NR = NR;
  l.rv = take((size_t)NR * 4);
  l.rt = take((size_t)NR * 4);
  l.ru = take((size_t)NR * 4);
  l.rk = take((size_t)NR * 8);
  l.lgn = take(ZP > 0 ? 33 * 8 : 0);
  l.bytes = o;
  l.H = H;
  return l;
}

// The staging kernel's shared memory for one position: the logits, each
// entry's hash slot, the hash table, and per branch row its largest logit
// (ordered) and fixed-point lse.
struct StageLayout {
  size_t lg, eu, hk, rmx, fl, bytes;
};
__host__ __device__ inline StageLayout stage_layout(int Z, int K, int H) {
  StageLayout l;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o += (bytes + 15) & ~(size_t)15;
    return at;
  };
  const size_t ZK = (size_t)Z * K;
  l.fl = take((size_t)Z * 8);
  l.lg = take(ZK * 4);
  l.hk = take((size_t)H * 4);
  l.eu = take(ZK * 2);
  l.rmx = take((size_t)Z * 4);
  l.bytes = o;
  return l;
}

// The dense width for Z branches (0: the sparse form only).
__host__ __device__ inline int dense_width(int Z) {
  return Z == 1 ? 1 : Z == 2 ? 2 : Z <= 4 ? 4 : Z <= 8 ? 8 : 0;
}

struct MixSm {
  const int64_t *flse, *fmax, *mq;
  const int64_t *lq;  // per entry: logit - lse in fixed point (kNegFix for a -inf logit)
  const float *C;
  const int *utok, *nu;
  const float *dE, *Ee;
  const int16_t *dR;
  const uint16_t *ue;
  int64_t *Pn, *Sn, *lrn;
  float *acc, *wz, *An;
  uint32_t *taken, *mask;
  int *par, *dep, *tok, *pu, *pt;  // pu, pt: the pending child's union index and token
  int Z, K, ZK, UW, W, b;
};

// The conversions below use 32-bit converts and integer shifts only: a
// conversion between a 64-bit integer and a float costs about a hundred
// cycles on this part, more than the rest of a pop step.

// round(x 2^40) for a logit x, as tb::fix_logit (clamped to 2^17; -inf and
// NaN give kNegFix), from the float's fields.
__device__ __forceinline__ int64_t fix_f32(float x) {
  if (!(x > -INFINITY)) return kNegFix;
  x = fminf(fmaxf(x, -tb::kMaxLogit), tb::kMaxLogit);
  const uint32_t bits = __float_as_uint(x);
  const int ex = (int)((bits >> 23) & 0xFFu);
  if (ex == 0) return 0;  // zero or subnormal: below 2^-126
  const int64_t m = (int64_t)((bits & 0x7FFFFFu) | 0x800000u);
  const int sh = ex - 127 - 23 + 40;  // x 2^40 = m 2^sh, sh <= 34
  int64_t v;
  if (sh >= 0) {
    v = m << sh;
  } else if (sh < -24) {
    v = 0;  // below 2^-1
  } else {  // round half to even
    const int r = -sh;
    const int64_t q = m >> r, rem = m & ((1ll << r) - 1), half = 1ll << (r - 1);
    v = q + ((rem > half || (rem == half && (q & 1))) ? 1 : 0);
  }
  return (bits >> 31) ? -v : v;
}

// exp(D 2^-40) for D <= 0: k = nearest integer to x / ln 2 from an estimate of
// x within 2^-8, f = D - k ln 2 exactly in fixed point (|f| < 0.36), result
// 2^k expf(f) with f rounded to 2^-31 first.
__device__ __forceinline__ float exp_fix(int64_t D0) {
  const int64_t D = D0 < kExpCut ? kExpCut : D0;
  const float xa = (float)(int)(D >> 32) * 0.00390625f;
  const int k = __float2int_rn(xa * 1.4426950408889634f);
  const int64_t f = D - (int64_t)k * kLn2Fix;
  const float ff = (float)(int)(f >> 9) * 4.656612873077393e-10f;
  const float r = ldexpf(expf(ff), k);
  return D0 < kExpCut ? 0.f : r;
}

// log(v) in 2^-40 units for a normal float v > 0: v = m 2^e with m in
// [2^-1/2, 2^1/2] from the float's fields, e ln 2 in fixed point, logf(m)
// (|logf(m)| < 0.35) rounded to 2^-30.
__device__ __forceinline__ int64_t log_fix(float v) {
  const uint32_t bits = __float_as_uint(v);
  int e = (int)(bits >> 23) - 127;
  float m = __uint_as_float((bits & 0x7FFFFFu) | 0x3F800000u);  // [1, 2)
  if (m > 1.41421356f) {
    m *= 0.5f;
    ++e;
  }
  return (int64_t)e * kLn2Fix + ((int64_t)__float2int_rn(logf(m) * 1073741824.f) << 10);
}

__device__ __forceinline__ int64_t warp_max_i64(int64_t x) {
  const uint64_t k = tb::key_of(x);
  const uint32_t h = __reduce_max_sync(kFull, (uint32_t)(k >> 32));
  const uint32_t l = __reduce_max_sync(kFull, (uint32_t)(k >> 32) == h ? (uint32_t)k : 0u);
  return (int64_t)((((uint64_t)h << 32) | l) ^ 0x8000000000000000ull);
}

struct Pick {
  float v;     // the best untaken child's scaled rho (0: none with a positive sum)
  int t, u;    // its token and union index
  bool any;    // some untaken child exists
};

// The warp's best of the lanes' (value desc, token asc) candidates.  A lane's
// candidates are distinct union tokens, so the winner is one lane's and its
// union index is the largest among lanes holding (value, token).
__device__ __forceinline__ Pick warp_pick(float bv, int bt, int bu, bool any) {
  const uint32_t vb = __float_as_uint(bv);  // bv >= 0: the bits order as the values
  const uint32_t m = __reduce_max_sync(kFull, vb);
  const int tm = __reduce_min_sync(kFull, vb == m ? bt : INT_MAX);
  Pick p;
  p.u = __reduce_max_sync(kFull, (vb == m && bt == tm) ? bu : -1);
  p.v = __uint_as_float(m);
  p.t = tm;
  p.any = __any_sync(kFull, any);
  return p;
}

// A lane's best (value desc, token asc) by value alone; the tokens are read
// only on an exact tie.
__device__ __forceinline__ void lane_track(float v, int u, const int *ut, float &bv, int &bu) {
  if (v > bv) {
    bv = v;
    bu = u;
  } else if (v == bv && v > 0.f && ut[u] < ut[bu]) {
    bu = u;
  }
}

// ---------------------------------------------------------------- dense form

template <int ZP>
__device__ __forceinline__ void load_e(const float *p, float (&e)[ZP]) {
  if constexpr (ZP == 1) {
    e[0] = p[0];
  } else if constexpr (ZP == 2) {
    const float2 v = *reinterpret_cast<const float2 *>(p);
    e[0] = v.x;
    e[1] = v.y;
  } else {
#pragma unroll
    for (int h = 0; h < ZP / 4; ++h) {
      const float4 v = reinterpret_cast<const float4 *>(p)[h];
      e[4 * h] = v.x;
      e[4 * h + 1] = v.y;
      e[4 * h + 2] = v.z;
      e[4 * h + 3] = v.w;
    }
  }
}

// This warp's part of the picks for node qa (row da, taken-bits apply) and
// for the new node qb (row db, nothing taken; qb = -1 for none): blocks
// c = warp, warp + 4, ... of 32 union tokens, lane l taking u = 32 c + l.
template <int ZP>
__device__ __forceinline__ void part_pick(const MixSm &s, int lane, int warp, int qa, int da,
                                          const float (&wa)[ZP], int qb, int db,
                                          const float (&wb)[ZP], Pick &pa, Pick &pb) {
  const int na = s.nu[da], nb = qb >= 0 ? s.nu[db] : 0, dbb = qb >= 0 ? db : 0;
  const float *Ea = s.dE + da * s.ZK * ZP, *Eb = s.dE + dbb * s.ZK * ZP;
  const uint32_t *tk = s.taken + qa * s.UW;
  const int *uta = s.utok + da * s.ZK, *utb = s.utok + dbb * s.ZK;
  float bva = 0.f, bvb = 0.f;
  int bua = -1, bub = -1;
  bool anya = false;
  const int nm = na > nb ? na : nb;
#pragma unroll 2
  for (int c = warp; c * 32 < nm; c += kPopWarps) {
    const int u = c * 32 + lane;
    float va = 0.f, vb = 0.f;
    uint32_t tw = 1u << lane;  // past the row: as if taken
    if (u < na) {
      float e[ZP];
      load_e<ZP>(Ea + u * ZP, e);
      tw = tk[c];
#pragma unroll
      for (int z = 0; z < ZP; ++z) va = fmaf(wa[z], e[z], va);
    }
    if (u < nb) {
      float e[ZP];
      load_e<ZP>(Eb + u * ZP, e);
#pragma unroll
      for (int z = 0; z < ZP; ++z) vb = fmaf(wb[z], e[z], vb);
    }
    if (!((tw >> lane) & 1u)) {
      anya = true;
      lane_track(va, u, uta, bva, bua);
    }
    if (u < nb) lane_track(vb, u, utb, bvb, bub);
  }
  const int bta = bua >= 0 ? uta[bua] : INT_MAX, btb = bub >= 0 ? utb[bub] : INT_MAX;
  pa = warp_pick(bva, bta, bua, anya);
  pb = warp_pick(bvb, btb, bub, nb > warp * 32);
}

// This warp's part of the pick for node q (row d, taken-bits apply).
template <int ZP>
__device__ __forceinline__ Pick part_pick1(const MixSm &s, int lane, int warp, int q, int d,
                                           const float (&w)[ZP]) {
  const int n = s.nu[d];
  const float *E = s.dE + d * s.ZK * ZP;
  const uint32_t *tk = s.taken + q * s.UW;
  const int *ut = s.utok + d * s.ZK;
  float bv = 0.f;
  int bu = -1;
  bool any = false;
#pragma unroll 2
  for (int c = warp; c * 32 < n; c += kPopWarps) {
    const int u = c * 32 + lane;
    float v = 0.f;
    uint32_t tw = 1u << lane;  // past the row: as if taken
    if (u < n) {
      float e[ZP];
      load_e<ZP>(E + u * ZP, e);
      tw = tk[c];
#pragma unroll
      for (int z = 0; z < ZP; ++z) v = fmaf(w[z], e[z], v);
    }
    if (!((tw >> lane) & 1u)) {
      any = true;
      lane_track(v, u, ut, bv, bu);
    }
  }
  return warp_pick(bv, bu >= 0 ? ut[bu] : INT_MAX, bu, any);
}

// A pick as the four warps exchange it.
struct Part {
  float v;
  int t, u, any;
};

// The best of the warps' parts: value, then token.
__device__ __forceinline__ Pick combine(const Part *pp) {
  Pick b;
  b.v = 0.f;
  b.t = INT_MAX;
  b.u = -1;
  b.any = false;
#pragma unroll
  for (int w = 0; w < kPopWarps; ++w) {
    const Part q = pp[w];
    b.any = b.any || q.any != 0;
    if (q.v > b.v || (q.v == b.v && q.v > 0.f && q.t < b.t)) {
      b.v = q.v;
      b.t = q.t;
      b.u = q.u;
    }
  }
  return b;
}

__device__ __forceinline__ void pop_barrier() {
  asm volatile("bar.sync 1, %0;" ::"r"(kPopWarps * 32) : "memory");
}

// Node q's children (row d) in the log domain: the largest branch term of
// each untaken child relative to S_q, in fixed point; then the sums rescaled
// by the largest of those, M.  Sets shift = M.
template <int ZP>
__device__ __forceinline__ Pick slow_dense(const MixSm &s, int lane, int q, int d, int64_t &shift) {
  const int Z = s.Z, K = s.K, n = s.nu[d];
  const int64_t Sq = s.Sn[q];
  int64_t base[ZP];
#pragma unroll
  for (int z = 0; z < ZP; ++z) {
    base[z] = kVeryNeg;
    if (z < Z) {
      const int64_t P = s.Pn[q * Z + z];
      if (P > kInfCut) base[z] = P - Sq;
    }
  }
  const int16_t *R = s.dR + (size_t)d * s.ZK * ZP;
  const uint32_t *tk = s.taken + q * s.UW;
  auto term = [&](int u, int z) -> int64_t {
    const int j = R[(size_t)u * ZP + z];
    if (j < 0 || base[z] == kVeryNeg) return kVeryNeg;
    const int64_t l = s.lq[(d * Z + z) * K + j];
    return l <= kInfCut ? kVeryNeg : base[z] + l;
  };
  int64_t best = kVeryNeg;
  for (int u = lane; u < n; u += 32) {
    if ((tk[u >> 5] >> lane) & 1u) continue;
#pragma unroll
    for (int z = 0; z < ZP; ++z) {
      const int64_t t = term(u, z);
      best = t > best ? t : best;
    }
  }
  const int64_t M = warp_max_i64(best);
  shift = M;
  float bv = 0.f;
  int bt = INT_MAX, bu = -1;
  bool any = false;
  if (M > kVeryNeg / 2) {
    const int *ut = s.utok + d * s.ZK;
    for (int u = lane; u < n; u += 32) {
      if ((tk[u >> 5] >> lane) & 1u) continue;
      any = true;
      float v = 0.f;
#pragma unroll
      for (int z = 0; z < ZP; ++z) {
        const int64_t t = term(u, z);
        if (t != kVeryNeg) {
          const int64_t D = t - M;
          v += exp_fix(D < 0 ? D : 0);
        }
      }
      lane_track(v, u, ut, bv, bu);
    }
    bt = bu >= 0 ? ut[bu] : INT_MAX;
  }
  return warp_pick(bv, bt, bu, any);
}

// P_z of node i, the child (union token u of row d - 1) of node p: lane z
// reads the token's rank in branch z.
template <int ZP>
__device__ __forceinline__ int64_t child_p_dense(const MixSm &s, int lane, int p, int d, int u) {
  const int z = lane < s.Z ? lane : 0;  // lanes past Z read branch 0 and drop it
  const int j = s.dR[((d - 1) * s.ZK + u) * ZP + z];
  const int64_t Pp = s.Pn[p * s.Z + z];
  const int64_t l = s.lq[((d - 1) * s.Z + z) * s.K + (j >= 0 ? j : 0)];
  int64_t P = Pp + l;
  P = P < kNegFix ? kNegFix : P;
  return (lane < s.Z && j >= 0 && Pp > kInfCut && l > kInfCut) ? P : kNegFix;
}

// --------------------------------------------------------------- sparse form

// The scaled sums of node q's children (row d) into acc[0..nu), one branch
// per pass.
__device__ __forceinline__ void scan_sparse(const MixSm &s, int lane, int q, int d, float *acc) {
  const int Z = s.Z, K = s.K, n = s.nu[d];
  for (int u = lane; u < n; u += 32) acc[u] = 0.f;
  __syncwarp();
  for (int z = 0; z < Z; ++z) {
    const float wv = s.wz[q * Z + z];
    if (wv == 0.f) continue;  // uniform over the warp
    const int e0 = (d * Z + z) * K;
    for (int j = lane; j < K; j += 32) {
      const int u = s.ue[e0 + j];
      acc[u] = fmaf(wv, s.Ee[e0 + j], acc[u]);
    }
    __syncwarp();
  }
}

__device__ __forceinline__ Pick pick_sparse(const MixSm &s, int lane, int q, int d, const float *acc) {
  const int n = s.nu[d];
  const uint32_t *tk = s.taken + q * s.UW;
  const int *ut = s.utok + d * s.ZK;
  float bv = 0.f;
  int bt = INT_MAX, bu = -1;
  bool any = false;
  for (int u = lane; u < n; u += 32) {
    if ((tk[u >> 5] >> lane) & 1u) continue;
    any = true;
    lane_track(acc[u], u, ut, bv, bu);
  }
  bt = bu >= 0 ? ut[bu] : INT_MAX;
  return warp_pick(bv, bt, bu, any);
}

__device__ __forceinline__ Pick slow_sparse(const MixSm &s, int lane, int q, int d, int64_t &shift) {
  const int Z = s.Z, K = s.K, n = s.nu[d];
  const int64_t Sq = s.Sn[q];
  int64_t *mx = reinterpret_cast<int64_t *>(s.acc);
  for (int u = lane; u < n; u += 32) mx[u] = kVeryNeg;
  __syncwarp();
  for (int z = 0; z < Z; ++z) {
    const int64_t P = s.Pn[q * Z + z];
    if (P <= kInfCut) continue;
    const int64_t base = P - Sq;
    const int e0 = (d * Z + z) * K;
    for (int j = lane; j < K; j += 32) {
      const int64_t l = s.lq[e0 + j];
      if (l <= kInfCut) continue;
      const int u = s.ue[e0 + j];
      const int64_t v = base + l;
      mx[u] = v > mx[u] ? v : mx[u];
    }
    __syncwarp();
  }
  const uint32_t *tk = s.taken + q * s.UW;
  int64_t best = kVeryNeg;
  for (int u = lane; u < n; u += 32)
    if (!((tk[u >> 5] >> lane) & 1u)) best = mx[u] > best ? mx[u] : best;
  const int64_t M = warp_max_i64(best);
  __syncwarp();
  shift = M;
  if (M <= kVeryNeg / 2) return warp_pick(0.f, INT_MAX, -1, false);
  float *acc = s.acc;
  for (int u = lane; u < n; u += 32) acc[u] = 0.f;
  __syncwarp();
  for (int z = 0; z < Z; ++z) {
    const int64_t P = s.Pn[q * Z + z];
    if (P <= kInfCut) continue;
    const int64_t base = P - Sq - M;
    const int e0 = (d * Z + z) * K;
    for (int j = lane; j < K; j += 32) {
      const int64_t l = s.lq[e0 + j];
      if (l <= kInfCut) continue;
      const int u = s.ue[e0 + j];
      const int64_t D = base + l;
      acc[u] += exp_fix(D < 0 ? D : 0);
    }
    __syncwarp();
  }
  return pick_sparse(s, lane, q, d, acc);
}

// P_z of node i, the child (union token u of row d - 1) of node p: a warp
// search of the row's entries for u.
__device__ __forceinline__ int64_t child_p_sparse(const MixSm &s, int lane, int p, int i, int d,
                                                  int u) {
  if (lane < s.Z) s.Pn[i * s.Z + lane] = kNegFix;
  __syncwarp();
  const int e0 = (d - 1) * s.ZK;
  for (int e = lane; e < s.ZK; e += 32) {
    if (s.ue[e0 + e] != u) continue;
    const int z = e / s.K;
    const int64_t Pp = s.Pn[p * s.Z + z], l = s.lq[e0 + e];
    int64_t v = kNegFix;
    if (Pp > kInfCut && l > kInfCut) {
      v = Pp + l;
      v = v < kNegFix ? kNegFix : v;
    }
    s.Pn[i * s.Z + z] = v;
  }
  __syncwarp();
  return lane < s.Z ? s.Pn[i * s.Z + lane] : kNegFix;
}

// ----------------------------------------------------------------- both forms

// The sparse form's pending children of node qa (row da) and of the new node
// qb (row db, or qb = -1), with the log-domain rescan of either where its
// best falls below 2^-100; shifts sa, sb of their keys.
__device__ __forceinline__ void pick_sparse2(const MixSm &s, int lane, int qa, int da, int qb, int db,
                                             Pick &pa, int64_t &sa, Pick &pb, int64_t &sb) {
  sa = sb = 0;
  pb.v = 0.f;
  pb.t = INT_MAX;
  pb.u = -1;
  pb.any = false;
  scan_sparse(s, lane, qa, da, s.acc);
  if (qb >= 0) scan_sparse(s, lane, qb, db, s.acc + s.ZK);
  pa = pick_sparse(s, lane, qa, da, s.acc);
  if (qb >= 0) pb = pick_sparse(s, lane, qb, db, s.acc + s.ZK);
  __syncwarp();
  if (pa.v < kTiny && pa.any) {
    pa = slow_sparse(s, lane, qa, da, sa);
    __syncwarp();
  }
  if (qb >= 0 && pb.v < kTiny && pb.any) {
    pb = slow_sparse(s, lane, qb, db, sb);
    __syncwarp();
  }
}

// The pending entry of node q (children at depth dchild) goes to lane q % 32,
// slot q / 32, as a 96-bit key: the order image of its score, then the tie
// word (bit 31: exact, below it 0x7FFFFFFF - (dchild << 16 | q)), so that among
// equal scores an exact entry comes before a bound (lazy) one, then lower depth
// and node.  An exact entry is the node's best untaken child; a lazy one an
// upper bound on all its children's scores.  A zero key: none.
__device__ __forceinline__ uint32_t tie_word(int q, int dchild, bool exact) {
  return (exact ? 0x80000000u : 0u) | (0x7FFFFFFFu - (((uint32_t)dchild << 16) | (uint32_t)q));
}
__device__ __forceinline__ void untie(uint32_t mt, int &q, int &dchild, bool &exact) {
  const uint32_t sec = 0x7FFFFFFFu - (mt & 0x7FFFFFFFu);
  q = (int)(sec & 0xFFFFu);
  dchild = (int)(sec >> 16);
  exact = (mt >> 31) != 0u;
}

template <int S>
struct Pending {
  uint32_t kh[S], kl[S], kt[S];  // the 96-bit key

  __device__ __forceinline__ void clear() {
#pragma unroll
    for (int i = 0; i < S; ++i) kh[i] = kl[i] = kt[i] = 0u;
  }
  __device__ __forceinline__ void set_key(int lane, int q, int dchild, bool ok, int64_t score,
                                          bool exact) {
    uint32_t hi = 0u, lo = 0u, tw = 0u;
    if (ok) {
      const uint64_t k = tb::key_of(score);
      hi = (uint32_t)(k >> 32);
      lo = (uint32_t)k;
      tw = tie_word(q, dchild, exact);
    }
    const int sl = q >> 5;
#pragma unroll
    for (int i = 0; i < S; ++i) {
      const bool me = lane == (q & 31) && i == sl;
      kh[i] = me ? hi : kh[i];
      kl[i] = me ? lo : kl[i];
      kt[i] = me ? tw : kt[i];
    }
  }
  // node q's best untaken child from a pick, exact; lane 0 records its union
  // index and token in this warp's copy
  __device__ __forceinline__ void set(const MixSm &s, int lane, int q, int dchild, const Pick &p,
                                      int64_t score) {
    set_key(lane, q, dchild, p.v > 0.f, score, true);
    if (lane == 0) {
      s.pu[q] = p.u;
      s.pt[q] = p.t;
    }
  }
  // The best key over the warp (all zero: none).
  __device__ __forceinline__ void best(uint32_t &mh, uint32_t &ml, uint32_t &mt) const {
    uint32_t bh = kh[0], bl = kl[0], bt = kt[0];
#pragma unroll
    for (int i = 1; i < S; ++i) {
      const bool g = tb::key_gt(kh[i], kl[i], kt[i], bh, bl, bt);
      bh = g ? kh[i] : bh;
      bl = g ? kl[i] : bl;
      bt = g ? kt[i] : bt;
    }
    tb::warp_best(bh, bl, bt, mh, ml, mt);
  }
};

// Staging: one CTA per (block position d + 1, request r) builds that
// position's tables in the workspace.  Work items are (branch row, 64-column
// block) pairs, one warp each, lane l taking columns j0 + l and j0 + 32 + l:
// (A) the logits and tokens, four items' loads in flight: logit - lse in
// fixed point, each token into the position's hash table (at most half
// full), the row's largest logit; (B) warp 0 numbers the table's used slots
// (lane l owns slots 32 q + l; numbered lane by lane after a warp scan), the
// union of the branches' tokens; (C) each entry's union index and
// E = exp(logit - its row's largest), scattered to its union token's record
// in the dense form.
template <int ZP>
__global__ void __launch_bounds__(kMixThreads) mixture_stage_kernel(MixArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int d = blockIdx.x, r = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int NW = kMixThreads / 32;
  const int Z = a.Z, b = a.b, K = a.K, ZK = Z * K;
  const MixLayout L = mix_layout(Z, b, K, a.n_max, ZP);
  const int H = L.H, hshift = 32 - (31 - __clz(H));
  const StageLayout SL = stage_layout(Z, K, H);
  float *lgs = reinterpret_cast<float *>(smem + SL.lg);
  int *hk = reinterpret_cast<int *>(smem + SL.hk);
  uint16_t *eu = reinterpret_cast<uint16_t *>(smem + SL.eu);
  uint32_t *rmx = reinterpret_cast<uint32_t *>(smem + SL.rmx);
  int64_t *fl = reinterpret_cast<int64_t *>(smem + SL.fl);
  unsigned char *w = a.ws + (size_t)r * a.ws_stride;
  int64_t *flse = reinterpret_cast<int64_t *>(w + L.flse) + d * Z;
  int64_t *fmax = reinterpret_cast<int64_t *>(w + L.fmax) + d * Z;
  int64_t *mq = reinterpret_cast<int64_t *>(w + L.mq) + d * Z;
  int64_t *lq = reinterpret_cast<int64_t *>(w + L.lq) + (size_t)d * ZK;
  int *utok = reinterpret_cast<int *>(w + L.utok) + (size_t)d * ZK;
  int *nu = reinterpret_cast<int *>(w + L.nu);
  uint16_t *ue = reinterpret_cast<uint16_t *>(w + L.ue) + (size_t)d * ZK;
  float *dE = reinterpret_cast<float *>(w + L.dE) + (size_t)d * ZK * ZP;
  int16_t *dR = reinterpret_cast<int16_t *>(w + L.dR) + (size_t)d * ZK * ZP;
  float *Ee = reinterpret_cast<float *>(w + L.ee) + (size_t)d * ZK;

  griddep_wait();
  griddep_launch_dependents();

  for (int q = tid; q < H; q += kMixThreads) hk[q] = kEmptySlot;
  for (int q = tid; q < Z; q += kMixThreads) {
    rmx[q] = 0u;  // below every ordered value
    const int64_t v = tb::fix_lse(__ldg(a.lse + ((size_t)r * Z + q) * b + d));
    fl[q] = v;
    flse[q] = v;
  }
  if constexpr (ZP > 0) {  // the position's union records cleared (E 0, rank -1)
    const int nq = ZK * ZP;
    if ((nq & 3) == 0 && ((uintptr_t)dE & 15) == 0 && ((uintptr_t)dR & 7) == 0) {
      for (int q = tid; q < nq / 4; q += kMixThreads) {
        reinterpret_cast<float4 *>(dE)[q] = make_float4(0.f, 0.f, 0.f, 0.f);
        reinterpret_cast<uint2 *>(dR)[q] = make_uint2(0xFFFFFFFFu, 0xFFFFFFFFu);
      }
    } else {
      for (int q = tid; q < nq; q += kMixThreads) {
        dE[q] = 0.f;
        dR[q] = -1;
      }
    }
  }
  __syncthreads();

  auto insert = [&](int tkn) -> uint16_t {
    uint32_t sl = ((uint32_t)tkn * 0x9E3779B1u) >> hshift;
    for (int it = 0; it < H; ++it) {
      const int old = atomicCAS(hk + sl, kEmptySlot, tkn);
      if (old == kEmptySlot || old == tkn) break;
      sl = (sl + 1) & (uint32_t)(H - 1);
    }
    return (uint16_t)sl;
  };
  const int KB = (K + 63) >> 6, items = Z * KB;
  const size_t rb = (size_t)r * Z * b * K;
  constexpr int UI = 4;
  for (int it0 = warp; it0 < items; it0 += NW * UI) {  // (A)
    float x[UI][2];
    int t[UI][2];
#pragma unroll
    for (int k = 0; k < UI; ++k) {
      const int item = it0 + k * NW;
      const int z = item / KB, j0 = (item - z * KB) << 6;
      const size_t g = rb + ((size_t)z * b + d) * K;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int j = j0 + 32 * h + lane;
        const bool ok = item < items && j < K;
        x[k][h] = ok ? __ldg(a.topk_logit + g + j) : -INFINITY;
        t[k][h] = ok ? __ldg(a.topk_tok + g + j) : 0;
      }
    }
#pragma unroll
    for (int k = 0; k < UI; ++k) {
      const int item = it0 + k * NW;
      if (item >= items) break;  // uniform over the warp
      const int z = item / KB, j0 = (item - z * KB) << 6;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int j = j0 + 32 * h + lane;
        if (j < K) {
          lgs[z * K + j] = x[k][h];
          const int64_t fx = fix_f32(x[k][h]);
          lq[z * K + j] = fx == kNegFix ? kNegFix : fx - fl[z];
          eu[z * K + j] = insert(t[k][h]);
        }
      }
      float mx = fmaxf(x[k][0], x[k][1]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
      if (lane == 0) atomicMax(rmx + z, ord_f32(mx));
    }
  }
  __syncthreads();
  if (warp == 0) {  // (B)
    const int S_ = H >> 5;
    int cnt = 0;
    for (int q = 0; q < S_; ++q) cnt += hk[32 * q + lane] != kEmptySlot;
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += v;
    }
    int u = incl - cnt;
    for (int q = 0; q < S_; ++q) {
      const int v = hk[32 * q + lane];
      if (v != kEmptySlot) {
        utok[u] = v;
        hk[32 * q + lane] = u++;
      }
    }
    if (lane == 31) nu[d] = incl;
  }
  __syncthreads();
  for (int item = warp; item < items; item += NW) {  // (C)
    const int z = item / KB, j0 = (item - z * KB) << 6;
    const int64_t fm = fix_f32(unord_f32(rmx[z]));
    if (lane == 0 && j0 == 0) {
      fmax[z] = fm;
      mq[z] = fm == kNegFix ? kNegFix : fm - fl[z];
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int j = j0 + 32 * h + lane;
      if (j < K) {
        const int e = z * K + j;
        int u = hk[eu[e]];
        u = (unsigned)u < (unsigned)ZK ? u : 0;  // (a token equal to INT32_MIN)
        const int64_t fx = fix_f32(lgs[e]);
        const float ev = (fm == kNegFix || fx == kNegFix) ? 0.f : exp_fix(fx - fm);
        ue[e] = (uint16_t)u;
        if constexpr (ZP > 0) {
          dE[u * ZP + z] = ev;
          dR[u * ZP + z] = (int16_t)j;
        } else {
          Ee[e] = ev;
        }
      }
    }
  }
}

// The pops of request r on its tables (copied from the workspace).
template <int S, int ZP>
__global__ void __launch_bounds__(kMixThreads, 1) build_tree_mixture_kernel(MixArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int r = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int Z = a.Z, b = a.b, K = a.K, n_max = a.n_max, ZK = Z * K;
  const MixLayout L = mix_layout(Z, b, K, n_max, ZP);
  const int64_t *flse = reinterpret_cast<const int64_t *>(smem + L.flse);
  const int64_t *fmax = reinterpret_cast<const int64_t *>(smem + L.fmax);
  const int64_t *mq = reinterpret_cast<const int64_t *>(smem + L.mq);
  const int64_t *lq = reinterpret_cast<const int64_t *>(smem + L.lq);
  const int *utok = reinterpret_cast<const int *>(smem + L.utok);
  const int *nu = reinterpret_cast<const int *>(smem + L.nu);
  const uint16_t *ue = reinterpret_cast<const uint16_t *>(smem + L.ue);
  const float *dE = reinterpret_cast<const float *>(smem + L.dE);
  const int16_t *dR = reinterpret_cast<const int16_t *>(smem + L.dR);
  const float *Ee = reinterpret_cast<const float *>(smem + L.ee);
  float *C = reinterpret_cast<float *>(smem + L.cost);

  griddep_wait();  // the staging kernel's tables are complete
  griddep_launch_dependents();

  // ---- the tables into shared memory (16-byte chunks, several in flight),
  // and the cost row
  {
    const uint4 *src = reinterpret_cast<const uint4 *>(a.ws + (size_t)r * a.ws_stride);
    uint4 *dst = reinterpret_cast<uint4 *>(smem);
    const int n16 = (int)(L.r1 >> 4);
    constexpr int UC = 8;
    for (int q0 = tid; q0 < n16; q0 += kMixThreads * UC) {
      uint4 v[UC];
#pragma unroll
      for (int k = 0; k < UC; ++k) {
        const int q = q0 + k * kMixThreads;
        if (q < n16) v[k] = __ldcg(src + q);
      }
#pragma unroll
      for (int k = 0; k < UC; ++k) {
        const int q = q0 + k * kMixThreads;
        if (q < n16) dst[q] = v[k];
      }
    }
  }
  const float *cr = a.cost + (a.cost_per_request ? (size_t)r * (n_max + 1) : 0);
  bool bad = false;
  for (int i = tid; i <= n_max; i += kMixThreads) {
    const float c = __ldg(cr + i);
    C[i] = c;
    if (i >= 1) bad |= !(c > 0.f) || isinf(c);
  }
  const bool bad_cost = __syncthreads_or(bad) != 0;

  MixSm s;
  s.flse = flse;
  s.fmax = fmax;
  s.mq = mq;
  s.lq = lq;
  s.C = C;
  s.utok = utok;
  s.nu = nu;
  s.dE = dE;
  s.dR = dR;
  s.Ee = Ee;
  s.ue = ue;
  s.Z = Z;
  s.K = K;
  s.ZK = ZK;
  s.UW = (ZK + 31) / 32;
  s.W = (n_max + 31) / 32;
  s.b = b;
  const int W = s.W, UW = s.UW;
  // this warp's copies of the node state (the dense form keeps one per pop warp)
  const int cw = ZP > 0 ? (warp < kPopWarps ? warp : 0) : 0;
  s.Pn = reinterpret_cast<int64_t *>(smem + L.pn) + (size_t)cw * n_max * Z;
  s.Sn = reinterpret_cast<int64_t *>(smem + L.sn) + (size_t)cw * n_max;
  s.wz = reinterpret_cast<float *>(smem + L.wz) + (size_t)cw * n_max * Z;
  s.lrn = reinterpret_cast<int64_t *>(smem + L.lrn);
  s.acc = reinterpret_cast<float *>(smem + L.acc);
  s.An = reinterpret_cast<float *>(smem + L.an);
  s.taken = reinterpret_cast<uint32_t *>(smem + L.taken);
  s.mask = reinterpret_cast<uint32_t *>(smem + L.mask);
  s.par = reinterpret_cast<int *>(smem + L.par);
  s.dep = reinterpret_cast<int *>(smem + L.dep);
  s.tok = reinterpret_cast<int *>(smem + L.tok);
  s.pu = reinterpret_cast<int *>(smem + L.pu) + (size_t)cw * n_max;
  s.pt = reinterpret_cast<int *>(smem + L.pt) + (size_t)cw * n_max;
  Part *part = reinterpret_cast<Part *>(smem + L.part);  // [2 phases][2 nodes][kPopWarps]

  if constexpr (ZP > 0) {  // every node's taken-bits cleared once
    for (int q = tid; q < n_max * UW; q += kMixThreads) s.taken[q] = 0u;
    __syncthreads();
  }
  constexpr int kRun = ZP > 0 ? kPopWarps : 1;  // the warps that run the pops
  if (warp >= kRun) return;

  // ---- the root: P_z = log pi_z (a weight that is negative or not finite
  // counts as 0 and sets the status bit)
  bool badw = false;
  int64_t P0 = kNegFix;
  if (lane < Z) {
    const double w = a.pi[(size_t)r * Z + lane];
    badw = !(w >= 0.0) || isinf(w);
    if (!badw && w > 0.0) P0 = tb::fix_lse(log(w));
  }
  if (__any_sync(kFull, badw) && warp == 0 && lane == 0) atomicOr(&a.status[r], BASTION_STATUS_BAD_WEIGHT);
  const int rec = kRun - 1;  // the warp that keeps the tree's records
  if (warp == rec && lane == 0) {
    s.par[0] = -1;
    s.dep[0] = 0;
    s.tok[0] = a.root_token[r];
    s.lrn[0] = 0;
    s.An[0] = 1.f;
  }
  if (warp == rec)
    for (int q = lane; q < W; q += 32) s.mask[q] = q == 0 ? 1u : 0u;

  Pending<S> pend;
  pend.clear();
  float A_hi = 1.f, A_lo = 0.f;  // A_hat with Kahan compensation
  int N = 1;

  if constexpr (ZP > 0) {
    // ==== dense form: four warps, identical decisions, a quarter of each scan.
    // A new node's entry starts as a bound on its children's scores (lazy)
    // and is scanned only if that bound wins a select; the root's children
    // are sorted once and taken in order.
    int ph = 0;
    float *rv = reinterpret_cast<float *>(smem + L.rv);
    int *rt = reinterpret_cast<int *>(smem + L.rt);
    int *ru = reinterpret_cast<int *>(smem + L.ru);
    int64_t *rk = reinterpret_cast<int64_t *>(smem + L.rk);
    int64_t *lgn = reinterpret_cast<int64_t *>(smem + L.lgn);  // log k, k = 1..32
    // node i's weights (lane z) and scale for its children at row d; false when
    // no child can have a finite score
    auto weights = [&](int i, int d, int64_t P, float &wl) -> bool {
      wl = 0.f;
      if (d >= b) return false;
      const int64_t m = s.mq[d * Z + (lane < Z ? lane : 0)];
      const int64_t X = (lane < Z && P > kInfCut && m > kInfCut) ? P + m : kVeryNeg;
      const int64_t Smax = warp_max_i64(X);
      if (Smax <= kInfCut) return false;
      wl = exp_fix(X - Smax);  // 0 for a -inf branch
      if (lane < Z) s.wz[i * Z + lane] = wl;
      if (lane == 0) s.Sn[i] = Smax;
      return true;
    };
    // node q's best untaken child (row d, its weights in lanes z: wl), over
    // the four warps, and its key
    auto scan = [&](int q, int d, float wl, Pick &pa, int64_t &ka) {
      float wa[ZP];
#pragma unroll
      for (int z = 0; z < ZP; ++z) wa[z] = __shfl_sync(kFull, wl, z);
      pa = part_pick1<ZP>(s, lane, warp, q, d, wa);
      Part *pp = part + ph * 2 * kPopWarps;
      if (lane == 0) pp[warp] = Part{pa.v, pa.t, pa.u, pa.any ? 1 : 0};
      pop_barrier();
      pa = combine(pp);
      ph ^= 1;
      int64_t sa = 0;
      if (pa.v < kTiny && pa.any) pa = slow_dense<ZP>(s, lane, q, d, sa);
      ka = pa.v > 0.f ? s.Sn[q] + sa + log_fix(pa.v) : 0;
    };
    // a new node i at depth d with P_z(i) in lane z: its lazy entry, the bound
    // S + log(number of finite branches) (every weight is at most 1 and every
    // E at most 1) plus a margin for rounding; no exponentials
    auto lazy = [&](int i, int d, int64_t P) {
      if (lane < Z) s.Pn[i * Z + lane] = P;
      bool ok = false;
      int64_t ub = 0;
      if (d < b) {
        const int64_t m = s.mq[d * Z + (lane < Z ? lane : 0)];
        const int64_t X = (lane < Z && P > kInfCut && m > kInfCut) ? P + m : kVeryNeg;
        const int64_t Smax = warp_max_i64(X);
        ok = Smax > kInfCut;
        const int nf = __popc(__ballot_sync(kFull, X > kInfCut));
        ub = Smax + lgn[nf > 0 ? nf : 1] + kBoundSlack;
      }
      pend.set_key(lane, i, d + 1, ok, ub, false);
    };

    // ---- the root: its weights, then its children's values sorted once
    if (warp == 0) lgn[lane + 1] = log_fix((float)(lane + 1));
    float wl0;
    if (lane < Z) s.Pn[lane] = P0;
    const bool root_kids = weights(0, 0, P0, wl0);
    pop_barrier();  // the log table before any warp reads it
    const int n0 = root_kids ? nu[0] : 0;
    bool root_sorted = root_kids && n0 <= L.NR;
    int rc = 0;  // the next root child in sorted order
    if (root_sorted) {
      float wa[ZP];
#pragma unroll
      for (int z = 0; z < ZP; ++z) wa[z] = __shfl_sync(kFull, wl0, z);
      const int NR = L.NR;
      for (int k = tid; k < NR; k += kPopWarps * 32) {
        float v = -1.f;  // the padding sorts last
        int t = INT_MAX;
        if (k < n0) {
          float e[ZP];
          load_e<ZP>(dE + k * ZP, e);
          v = 0.f;
#pragma unroll
          for (int z = 0; z < ZP; ++z) v = fmaf(wa[z], e[z], v);
          t = utok[k];
        }
        rv[k] = v;
        rt[k] = t;
        ru[k] = k;
      }
      pop_barrier();
      // bitonic sort by (value desc, token asc); tokens of one row are distinct
      for (int size = 2; size <= NR; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
          for (int k = tid; k < NR / 2; k += kPopWarps * 32) {
            const int lo = 2 * k - (k & (stride - 1)), hi = lo + stride;
            const bool desc = (lo & size) == 0;
            const float va = rv[lo], vb = rv[hi];
            const int ta = rt[lo], tb = rt[hi];
            const bool b_first = vb > va || (vb == va && tb < ta);
            if (b_first == desc) {
              rv[lo] = vb;
              rv[hi] = va;
              rt[lo] = tb;
              rt[hi] = ta;
              const int x = ru[lo];
              ru[lo] = ru[hi];
              ru[hi] = x;
            }
          }
          pop_barrier();
        }
      }
      for (int k = tid; k < n0; k += kPopWarps * 32)
        rk[k] = rv[k] >= kTiny ? s.Sn[0] + log_fix(rv[k]) : 0;
      pop_barrier();
      const bool ok = n0 > 0 && rv[0] >= kTiny;
      if (ok) {
        pend.set_key(lane, 0, 1, true, rk[0], true);
      } else if (n0 > 0) {  // the largest child is tiny: the root is scanned as any node
        root_sorted = false;
        pend.set_key(lane, 0, 1, true, s.Sn[0] + lgn[Z] + kBoundSlack, false);
      }
    } else if (root_kids) {
      pend.set_key(lane, 0, 1, true, s.Sn[0] + lgn[Z] + kBoundSlack, false);
    }
    __syncwarp();

    while (N < n_max) {
      uint32_t mh, ml, mt;
      pend.best(mh, ml, mt);
      if ((mh | ml | mt) == 0u) break;  // no candidate left
      const int64_t sc = (int64_t)((((uint64_t)mh << 32) | ml) ^ 0x8000000000000000ull);
      if (sc < kInfCut) break;  // the best candidate has rho = 0
      int p, d;
      bool exact;
      untie(mt, p, d, exact);
      if (!exact) {
        // a bound won: node p's best untaken child replaces it, then select again
        float wl;
        const int64_t Pp = s.Pn[p * Z + (lane < Z ? lane : 0)];
        Pick pa;
        int64_t ka = 0;
        pa.v = 0.f;
        pa.t = INT_MAX;
        pa.u = -1;
        pa.any = false;
        if (weights(p, d - 1, lane < Z ? Pp : kNegFix, wl)) {
          __syncwarp();
          scan(p, d - 1, wl, pa, ka);
        }
        pend.set(s, lane, p, d, pa, ka);
        if (p == 0) root_sorted = false;
        __syncwarp();
        continue;
      }
      const float rho = exp_fix(sc);
      const bool from_list = p == 0 && root_sorted;
      const int u = from_list ? ru[rc] : s.pu[p], t = from_list ? rt[rc] : s.pt[p];
      const float Cp = C[N], Cn = C[N + 1];
      if (rho * Cp < (A_hi + A_lo) * (Cn - Cp)) break;  // S would decrease: keep T_N
      {
        const float y = rho - A_lo;
        const float tt = A_hi + y;
        A_lo = (tt - A_hi) - y;
        A_hi = tt;
      }
      const int i = N;
      N = i + 1;
      if (warp == kPopWarps - 1) {  // the lightest scanner keeps the tree's records
        if (lane == 0) {
          s.par[i] = p;
          s.dep[i] = d;
          s.tok[i] = t;
          s.lrn[i] = sc;
          s.An[i] = A_hi + A_lo;
        }
        if (lane < W) s.mask[i * W + lane] = s.mask[p * W + lane] | (lane == (i >> 5) ? (1u << (i & 31)) : 0u);
      }
      // the word of the taken child belongs to warp (u / 32) % 4
      if (lane == 0 && ((u >> 5) & (kPopWarps - 1)) == warp) s.taken[p * UW + (u >> 5)] |= 1u << (u & 31);
      lazy(i, d, child_p_dense<ZP>(s, lane, p, d, u));
      if (from_list) {  // the root's next child in sorted order
        ++rc;
        if (rc < n0 && rv[rc] >= kTiny) {
          pend.set_key(lane, 0, 1, true, rk[rc], true);
        } else if (rc < n0) {  // the rest are tiny: a bound (the score just taken), then a scan
          root_sorted = false;
          pend.set_key(lane, 0, 1, true, sc, false);
        } else {
          pend.set_key(lane, 0, 1, false, 0, true);
        }
      } else {  // the parent's next-best child
        __syncwarp();
        Pick pa;
        int64_t ka;
        scan(p, d - 1, lane < Z ? s.wz[p * Z + lane] : 0.f, pa, ka);
        pend.set(s, lane, p, d, pa, ka);
      }
      __syncwarp();  // lane 0's records before the next pop reads them
    }
  } else {
    // ==== sparse form: warp 0 alone
    if (lane < Z) s.Pn[lane] = P0;
    for (int q = lane; q < UW; q += 32) s.taken[q] = 0u;
    __syncwarp();
    auto setup = [&](int i, int d, int64_t P) -> bool {
      if (lane < Z) s.Pn[i * Z + lane] = P;
      if (d >= b) return false;
      const int64_t m = lane < Z ? s.mq[d * Z + lane] : kNegFix;
      const int64_t X = (lane < Z && P > kInfCut && m > kInfCut) ? P + m : kVeryNeg;
      const int64_t Smax = warp_max_i64(X);
      if (Smax <= kInfCut) return false;
      if (lane < Z) s.wz[i * Z + lane] = X <= kInfCut ? 0.f : exp_fix(X - Smax);
      for (int q = lane; q < UW; q += 32) s.taken[i * UW + q] = 0u;
      if (lane == 0) s.Sn[i] = Smax;
      return true;
    };
    auto keyed = [&](int qa, int da, int qb, int db, Pick &pa, int64_t &ka, Pick &pb, int64_t &kb) {
      __syncwarp();
      int64_t sa, sb;
      pick_sparse2(s, lane, qa, da, qb, db, pa, sa, pb, sb);
      ka = pa.v > 0.f ? s.Sn[qa] + sa + log_fix(pa.v) : 0;
      kb = (qb >= 0 && pb.v > 0.f) ? s.Sn[qb] + sb + log_fix(pb.v) : 0;
      __syncwarp();
    };
    if (setup(0, 0, P0)) {
      Pick pa, pb;
      int64_t ka, kb;
      keyed(0, 0, -1, 0, pa, ka, pb, kb);
      pend.set(s, lane, 0, 1, pa, ka);
      __syncwarp();
    }
    while (N < n_max) {
      uint32_t mh, ml, mt;
      pend.best(mh, ml, mt);
      if ((mh | ml | mt) == 0u) break;
      const int64_t sc = (int64_t)((((uint64_t)mh << 32) | ml) ^ 0x8000000000000000ull);
      if (sc < kInfCut) break;
      int p, d;
      bool exact;
      untie(mt, p, d, exact);
      const float rho = exp_fix(sc);
      const float Cp = C[N], Cn = C[N + 1];
      if (rho * Cp < (A_hi + A_lo) * (Cn - Cp)) break;
      {
        const float y = rho - A_lo;
        const float t = A_hi + y;
        A_lo = (t - A_hi) - y;
        A_hi = t;
      }
      const int i = N;
      N = i + 1;
      const int u = s.pu[p], t = s.pt[p];
      if (lane == 0) {
        s.par[i] = p;
        s.dep[i] = d;
        s.tok[i] = t;
        s.lrn[i] = sc;
        s.An[i] = A_hi + A_lo;
        s.taken[p * UW + (u >> 5)] |= 1u << (u & 31);
      }
      for (int q = lane; q < W; q += 32)
        s.mask[i * W + q] = s.mask[p * W + q] | (q == (i >> 5) ? (1u << (i & 31)) : 0u);
      const bool kids = setup(i, d, child_p_sparse(s, lane, p, i, d, u));
      Pick pa, pb;
      int64_t ka, kb;
      keyed(p, d - 1, kids ? i : -1, d, pa, ka, pb, kb);
      pend.set(s, lane, p, d, pa, ka);
      if (kids) pend.set(s, lane, i, d + 1, pb, kb);
      __syncwarp();  // lane 0's records before the next pop reads them
    }
  }
  if (warp != rec) return;
  __syncwarp();

  // ---- outputs
  const size_t nb = (size_t)r * n_max;
  const int ctx = a.ctx_len[r];
  const float L_ar = a.l_ar[r];
  if (lane == 0) {
    a.n_nodes[r] = N;
    if (bad_cost) atomicOr(&a.status[r], BASTION_STATUS_BAD_COST);
  }
  for (int i = lane; i < N; i += 32) {
    const size_t o = nb + i;
    const float Ah = s.An[i];
    a.parent[o] = s.par[i];
    a.depth[o] = s.dep[i];
    a.pos_id[o] = ctx + s.dep[i];
    a.token[o] = s.tok[i];
    a.log_rho[o] = __ll2float_rn(s.lrn[i]) * tb::kUnfix;
    a.a_hat[o] = Ah;
    a.speedup[o] = Ah * L_ar / C[i + 1];
  }
  for (int q = lane; q < N * W; q += 32) a.anc_mask[nb * W + q] = s.mask[q];
}

constexpr size_t kSmemCap = 227 * 1024;

}  // namespace

// The dense form's width when its tables fit in shared memory, else 0 (the
// sparse form).
int mixture_tree_form(int Z, int b, int K, int n_max) {
  const int zp = dense_width(Z);
  if (zp > 0 && mix_layout(Z, b, K, n_max, zp).bytes <= kSmemCap) return zp;
  return 0;
}

size_t mixture_tree_smem_bytes(int Z, int b, int K, int n_max) {
  return mix_layout(Z, b, K, n_max, mixture_tree_form(Z, b, K, n_max)).bytes;
}

// Workspace bytes of one request's tables (a multiple of 256).
size_t mixture_tree_ws_stride(int Z, int b, int K, int n_max) {
  return (mix_layout(Z, b, K, n_max, mixture_tree_form(Z, b, K, n_max)).r1 + 255) & ~(size_t)255;
}

int launch_build_tree_mixture(const float *topk_logit, const int32_t *topk_tok, const double *lse,
                              const double *pi, int B, int Z, int b, int K, int n_max,
                              const int32_t *root_token, const int32_t *ctx_len,
                              const float *cost_ms, int cost_per_request, const float *l_ar,
                              int32_t *n_nodes, int32_t *parent, int32_t *depth, int32_t *pos_id,
                              int32_t *token, float *log_rho, float *a_hat, float *speedup,
                              uint32_t *anc_mask, void *workspace, int32_t *status,
                              cudaStream_t stream) {
  MixArgs a;
  a.ws = static_cast<unsigned char *>(workspace);
  a.ws_stride = mixture_tree_ws_stride(Z, b, K, n_max);
  a.topk_logit = topk_logit;
  a.topk_tok = topk_tok;
  a.lse = lse;
  a.pi = pi;
  a.B = B;
  a.Z = Z;
  a.b = b;
  a.K = K;
  a.n_max = n_max;
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
  const int zp = mixture_tree_form(Z, b, K, n_max);
  const MixLayout ml = mix_layout(Z, b, K, n_max, zp);
  const size_t smem = ml.bytes, stage_smem = stage_layout(Z, K, ml.H).bytes;
  const int slots = tb::tree_slots(n_max);
  // the staging kernel: one CTA per (position, request)
  auto stage = [&](auto kern) {
    if (stage_smem > 48 * 1024 &&
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)stage_smem) !=
            cudaSuccess)
      return cudaErrorInvalidValue;
    return launch_pdl(kern, dim3(b, B), dim3(kMixThreads), stage_smem, stream, a);
  };
  const cudaError_t e0 = zp == 1   ? stage(mixture_stage_kernel<1>)
                         : zp == 2 ? stage(mixture_stage_kernel<2>)
                         : zp == 4 ? stage(mixture_stage_kernel<4>)
                         : zp == 8 ? stage(mixture_stage_kernel<8>)
                                   : stage(mixture_stage_kernel<0>);
  if (e0 != cudaSuccess) {
    cudaGetLastError();
    return BASTION_ERR_LAUNCH;
  }
  auto go = [&](auto kern) {
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return cudaErrorInvalidValue;
    return launch_pdl(kern, dim3(B), dim3(kMixThreads), smem, stream, a);
  };
  auto by_slots = [&](auto k1, auto k2, auto k4, auto k8) {
    return slots == 1 ? go(k1) : slots == 2 ? go(k2) : slots == 4 ? go(k4) : go(k8);
  };
#define BASTION_MIX_KERNELS(ZP_)                                                                 \
  by_slots(build_tree_mixture_kernel<1, ZP_>, build_tree_mixture_kernel<2, ZP_>,                 \
           build_tree_mixture_kernel<4, ZP_>, build_tree_mixture_kernel<8, ZP_>)
  const cudaError_t e = zp == 1   ? BASTION_MIX_KERNELS(1)
                        : zp == 2 ? BASTION_MIX_KERNELS(2)
                        : zp == 4 ? BASTION_MIX_KERNELS(4)
                        : zp == 8 ? BASTION_MIX_KERNELS(8)
                                  : BASTION_MIX_KERNELS(0);
#undef BASTION_MIX_KERNELS
  if (e != cudaSuccess) {
    cudaGetLastError();
    return BASTION_ERR_LAUNCH;
  }
  return cudaGetLastError() == cudaSuccess ? BASTION_OK : BASTION_ERR_LAUNCH;
}

}  // namespace bastion
