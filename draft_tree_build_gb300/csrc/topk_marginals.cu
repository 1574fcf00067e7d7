// Step 1 of the draft-tree path: softmax + top-K marginals over the full vocab.
//
// Bastion (gist.science/nl/paper/2605.29727), Methodologie §1: the block-
// diffusion drafter emits position-wise marginals q_k = softmax(l_k); the
// children of a depth-(k-1) tree node are the ranked tokens of q_k.
//
// Design (HBM-bound, one read of every logit):
//  * one thread-block cluster of CS CTAs per row (CS <= 8; 16 for the widest
//    rows).  CTA r stages slice r of the row in shared memory with one TMA
//    bulk copy (cp.async.bulk);
//  * pass A, per thread: the max of each of its 16-byte vectors (kept in
//    registers) and the thread max m_t.  Every CTA sends the 16-bit prefixes
//    of its 256 thread maxima' order keys to every CTA of the cluster with
//    asynchronous distributed-shared-memory stores (st.async), counted on the
//    receiver's mbarrier; while they travel it sums exp(l - m_t) over its
//    elements, one packed f32x2 FMA per two exponents and ex2 (the rounding
//    of m_t log2(e) is a common factor of the thread's terms, removed once);
//  * the row threshold T: from its copy of the row's CS*256 prefixes, every
//    CTA finds the K-th largest with one histogram of distances below the
//    largest.  T is the smallest float with the K-th largest prefix, so at
//    least K elements of the row reach it and the row's top K lies among the
//    elements >= T (on logit rows, K plus a few);
//  * pass B: the slice's elements >= T go to a list in shared memory as
//    64-bit keys (value desc, token asc); the CTA then sends the list
//    (zero-padded to a fixed length) and its (max, two-float sum of
//    exp(l - max), count) to the cluster's leader with asynchronous stores
//    counted on the leader's mbarrier, and exits;
//  * the leader waits for the row, ranks its keys by counting (the keys are
//    unique), writes the top K and lse = M + log(sum).  If a CTA's list
//    overflows (long runs of equal values), it selects the row's top K
//    exactly with a radix select over the row in global memory.
// Rows too wide for 16 slices, and K > 256, take the exact path in a kernel
// of their own.
#include <cuda_bf16.h>

#include <cstdlib>
#include <cstring>

#include "common.cuh"

namespace bastion {

namespace {

constexpr int kT = 256;      // threads per CTA (8 warps)
constexpr int kMaxCS = 16;   // CTAs per row at most
constexpr float kL2e = 1.4426950216293335f;       // log2(e) rounded to float
constexpr float kL2eLo = 1.925963033500011e-08f;  // log2(e) - kL2e
constexpr double kLn2 = 0.6931471805599453;       // ln 2

struct TopkArgs {
  const unsigned char *logits;
  int rows, b, V, K, CS, SL, seg, tab_bytes, body_bytes;
  int nst;  // stream path: stages of the widest row (its shared-memory layout)
  int64_t ld;  // elements
  float *topk_logq, *topk_logit;
  int32_t *topk_tok;
  double *lse;
  int32_t *status;
};

// One CTA's share of a row: its max, its two-float sum of exp(l - max) and
// the number of its keys >= T (16 bytes: one asynchronous store).
struct __align__(16) Part {
  float m, sx, sy;
  uint32_t n;
};

struct Scratch {
  uint32_t hist1[256];
  uint32_t red_u[8];
  float red_f[8];
  float2 red_s[8];
  Part part[kMaxCS];      // leader: each CTA's (max, sum, key count)
  int off[kMaxCS + 1];    // leader: where each CTA's keys go in the row list
  uint32_t n_loc;         // keys in this CTA's list (may pass seg: overflow)
  uint32_t n_exact;
  uint32_t n_hit;         // stream path: stages to read again
  uint32_t digit_info[2];
  int warp_tot[8];
  double lse;
};
constexpr int kScratchBytes = (int)((sizeof(Scratch) + 127) / 128 * 128);

// --------------------------------------------------------------------------- arithmetic
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 2^(x_i log2(e) - c) for four elements, summed in pairs: one packed f32x2
// FMA per two elements, then ex2.  With c = the float nearest m log2(e), the
// exponent is (x_i - m) log2(e) + (m log2(e) - c): every term of one thread
// carries the same factor 2^(m log2(e) - c), removed from the thread's sum
// once (see the callers).
__device__ __forceinline__ void exp4(float x0, float x1, float x2, float x3, float nc, float &s0,
                                     float &s1) {
  float t0, t1, t2, t3;
  asm("{\n .reg .b64 d, e, k, c;\n"
      " mov.b64 d, {%4, %5};\n mov.b64 e, {%6, %7};\n mov.b64 k, {%9, %9};\n"
      " mov.b64 c, {%8, %8};\n fma.rn.f32x2 d, d, k, c;\n fma.rn.f32x2 e, e, k, c;\n"
      " mov.b64 {%0, %1}, d;\n mov.b64 {%2, %3}, e;\n}\n"
      : "=f"(t0), "=f"(t1), "=f"(t2), "=f"(t3)
      : "f"(x0), "f"(x1), "f"(x2), "f"(x3), "f"(nc), "f"(kL2e));
  const float e0 = ex2(t0), e1 = ex2(t1), e2 = ex2(t2), e3 = ex2(t3);
  asm("{\n .reg .b64 a, c;\n mov.b64 a, {%2, %3};\n mov.b64 c, {%4, %5};\n"
      " add.rn.f32x2 a, a, c;\n mov.b64 {%0, %1}, a;\n}\n"
      : "=f"(s0), "=f"(s1)
      : "f"(e0), "f"(e1), "f"(e2), "f"(e3));
}

__device__ __forceinline__ float exp_shifted(float d) { return ex2(fmaf(d, kL2e, d * kL2eLo)); }

// Two-float sums: value = hi + lo.
__device__ __forceinline__ float2 two_sum(float a, float b) {
  const float s = a + b;
  const float bb = s - a;
  return make_float2(s, (a - (s - bb)) + (b - bb));
}
__device__ __forceinline__ float2 ff_add(float2 a, float2 b) {
  float2 s = two_sum(a.x, b.x);
  s.y += a.y + b.y;
  return two_sum(s.x, s.y);
}
__device__ __forceinline__ float2 ff_warp_sum(float2 v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float2 w = make_float2(__shfl_xor_sync(kFull, v.x, o), __shfl_xor_sync(kFull, v.y, o));
    v = ff_add(v, w);
  }
  return v;
}

template <int ES>
__device__ __forceinline__ float load_elem(const unsigned char *p) {
  if constexpr (ES == 4) {
    return *reinterpret_cast<const float *>(p);
  } else {
    return __uint_as_float((uint32_t)(*reinterpret_cast<const uint16_t *>(p)) << 16);
  }
}

template <int ES>
__device__ __forceinline__ void unpack(const uint4 &x, float (&f)[16 / ES]) {
  if constexpr (ES == 4) {
    f[0] = __uint_as_float(x.x); f[1] = __uint_as_float(x.y);
    f[2] = __uint_as_float(x.z); f[3] = __uint_as_float(x.w);
  } else {
    f[0] = bf16lo(x.x); f[1] = bf16hi(x.x); f[2] = bf16lo(x.y); f[3] = bf16hi(x.y);
    f[4] = bf16lo(x.z); f[5] = bf16hi(x.z); f[6] = bf16lo(x.w); f[7] = bf16hi(x.w);
  }
}

template <int ES>
__device__ __forceinline__ float vmax(const uint4 &x) {
  if constexpr (ES == 4) {
    return fmaxf(fmaxf(__uint_as_float(x.x), __uint_as_float(x.y)),
                 fmaxf(__uint_as_float(x.z), __uint_as_float(x.w)));
  } else {
    uint32_t a, c, m;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(a) : "r"(x.x), "r"(x.y));
    asm("max.bf16x2 %0, %1, %2;" : "=r"(c) : "r"(x.z), "r"(x.w));
    asm("max.bf16x2 %0, %1, %2;" : "=r"(m) : "r"(a), "r"(c));
    return fmaxf(bf16lo(m), bf16hi(m));
  }
}

// Sum of 2^(x log2(e) + nc) over one 16-byte vector.
template <int ES>
__device__ __forceinline__ float vexp_sum(const uint4 &x, float nc) {
  float f[16 / ES];
  unpack<ES>(x, f);
  if constexpr (ES == 2) {
    float p0, p1, q0, q1;
    exp4(f[0], f[1], f[2], f[3], nc, p0, p1);
    exp4(f[4], f[5], f[6], f[7], nc, q0, q1);
    return (p0 + p1) + (q0 + q1);
  } else {
    float p0, p1;
    exp4(f[0], f[1], f[2], f[3], nc, p0, p1);
    return p0 + p1;
  }
}

// --------------------------------------------------------------------------- selection helpers
// Warp 0: scanning the 256 bins of h from 255 down, the bin at which the
// running count reaches need (0 < need <= total), and the count above it,
// into info[0], info[1].
__device__ __forceinline__ void find_digit(const uint32_t *h, uint32_t need, uint32_t *info,
                                           int lane) {
  uint32_t cnt[8], tot = 0;
#pragma unroll
  for (int q = 0; q < 8; ++q) { cnt[q] = h[255 - 8 * lane - q]; tot += cnt[q]; }
  uint32_t incl = tot;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += y;
  }
  const uint32_t above = incl - tot;
  if (above < need && incl >= need) {
    uint32_t run = above;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      if (run + cnt[q] >= need) {
        info[0] = 255u - 8u * lane - q;
        info[1] = run;
        break;
      }
      run += cnt[q];
    }
  }
}

// Adds 1 to h[bin] for every lane whose bin is < 256 (one atomic per distinct
// bin of the warp).  All lanes call it.
__device__ __forceinline__ void hist_add(uint32_t *h, uint32_t bin, int lane) {
  const uint32_t peers = __match_any_sync(kFull, bin);
  if (bin < 256u && lane == __ffs(peers) - 1) atomicAdd(&h[bin], (uint32_t)__popc(peers));
}

// Exclusive prefix sum over the CTA of one int per thread.
__device__ __forceinline__ int cta_exclusive_scan(int x, Scratch &sc) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) sc.warp_tot[warp] = incl;
  __syncthreads();
  int before = 0;
  for (int w = 0; w < warp; ++w) before += sc.warp_tot[w];
  __syncthreads();
  return before + incl - x;
}

// The row's top min(K, V) keys, exactly and unsorted, into dst: a radix select
// of the K-th largest order key (8-bit digits) over the row in global memory,
// then every element above it and the lowest-token elements equal to it.  All
// threads of the CTA call it; returns the number of keys written.
template <int ES>
__device__ int row_topk_exact(const unsigned char *g, int V, int K, uint64_t *dst, Scratch &sc) {
  const int tid = threadIdx.x, lane = tid & 31;
  const int want = min(K, V);
  int kk = want;
  uint32_t prefix = 0, pmask = 0;
  for (int shift = 24; shift >= 0; shift -= 8) {
    sc.hist1[tid] = 0u;
    __syncthreads();
    for (int e = tid; e < V; e += kT) {
      const uint32_t o = ord_f32(load_elem<ES>(g + (size_t)e * ES));
      if ((o & pmask) == prefix) atomicAdd(&sc.hist1[(o >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (tid < 32) find_digit(sc.hist1, (uint32_t)kk, sc.digit_info, lane);
    __syncthreads();
    prefix |= sc.digit_info[0] << shift;
    pmask |= 255u << shift;
    kk -= (int)sc.digit_info[1];
  }
  // kk elements equal to the threshold key are taken, lowest tokens first
  const int per = (V + kT - 1) / kT;
  const int lo = min(V, tid * per), hi = min(V, lo + per);
  int eq = 0;
  for (int e = lo; e < hi; ++e) eq += ord_f32(load_elem<ES>(g + (size_t)e * ES)) == prefix;
  int rank_eq = cta_exclusive_scan(eq, sc);
  if (tid == 0) sc.n_exact = 0u;
  __syncthreads();
  for (int e = lo; e < hi; ++e) {
    const float v = load_elem<ES>(g + (size_t)e * ES);
    const uint32_t o = ord_f32(v);
    bool take = o > prefix;
    if (o == prefix) take = rank_eq++ < kk;
    if (take) dst[atomicAdd(&sc.n_exact, 1u)] = make_key(v, (uint32_t)e);
  }
  __syncthreads();
  return want;
}

// Ranks n unique keys of list by counting, writes the top K's logits and
// tokens and keeps each key's rank in rk (all threads call it; list[n] must be
// readable and zero when n is odd).  Four lanes count for one key, each over
// a quarter of the list.
__device__ __forceinline__ void rank_keys(const TopkArgs &a, int row, const uint64_t *list, int n,
                                          int *rk) {
  const int K = a.K, sub = threadIdx.x & 3;
  const ulonglong2 *l2 = reinterpret_cast<const ulonglong2 *>(list);
  const int n2 = (n + 1) >> 1;
  const int end = (n + kT / 4 - 1) / (kT / 4) * (kT / 4);  // the same trip count for a warp's lanes
  for (int i = threadIdx.x >> 2; i < end; i += kT / 4) {
    const uint64_t key = i < n ? list[i] : ~0ull;
    int r = 0;
#pragma unroll 4
    for (int j = sub; j < n2; j += 4) {
      const ulonglong2 p = l2[j];
      r += (p.x > key) + (p.y > key);
    }
    r += __shfl_xor_sync(kFull, r, 1);
    r += __shfl_xor_sync(kFull, r, 2);
    if (sub == 0 && i < n) {
      rk[i] = r;
      if (r < K) {
        const size_t o = (size_t)row * K + r;
        a.topk_logit[o] = key_value(key);
        a.topk_tok[o] = (int32_t)key_token(key);
      }
    }
  }
}

// log q = logit - lse for the ranked keys (after rank_keys and a barrier).
__device__ __forceinline__ void write_logq(const TopkArgs &a, int row, const uint64_t *list, int n,
                                           const int *rk, double lse) {
  if (!a.topk_logq) return;
  for (int i = threadIdx.x; i < n; i += kT) {
    const int r = rk[i];
    if (r < a.K) a.topk_logq[(size_t)row * a.K + r] = (float)((double)key_value(list[i]) - lse);
  }
}

// --------------------------------------------------------------------------- slice geometry
struct Slice {
  int e0, n, nh, t0, nvec, body;  // body: bytes of the 16-byte aligned middle
  const unsigned char *g0;
  uintptr_t ga0;
};

template <int ES>
__device__ __forceinline__ Slice slice_at(const TopkArgs &a, int row, int r) {
  Slice s;
  s.e0 = r * a.SL;
  s.n = max(0, min(a.V - s.e0, a.SL));
  s.g0 = a.logits + ((size_t)row * (size_t)a.ld + (size_t)s.e0) * ES;
  s.ga0 = ((uintptr_t)s.g0 + 15) & ~(uintptr_t)15;
  const uintptr_t ga1 = ((uintptr_t)s.g0 + (uintptr_t)s.n * ES) & ~(uintptr_t)15;
  s.body = ga1 > s.ga0 ? (int)(ga1 - s.ga0) : 0;
  const int h = s.body ? (int)(s.ga0 - (uintptr_t)s.g0) : s.n * ES;
  s.nh = h / ES;
  s.t0 = (h + s.body) / ES;
  s.nvec = s.body / 16;
  return s;
}

// lse of the row from per-CTA (max, two-float sum) pairs; sets status bits.
__device__ __forceinline__ double row_lse(const TopkArgs &a, int row, const Part *pt, int n) {
  float M = -INFINITY;
  for (int q = 0; q < n; ++q) M = fmaxf(M, pt[q].m);
  float2 acc = make_float2(0.f, 0.f);
  for (int q = 0; q < n; ++q) {
    if (pt[q].m == -INFINITY) continue;
    const float e = expf(pt[q].m - M);
    const float ph = pt[q].sx * e;
    const float pl = fmaf(pt[q].sx, e, -ph) + pt[q].sy * e;
    acc = ff_add(acc, make_float2(ph, pl));
  }
  const double s = (double)acc.x + (double)acc.y;
  // log s = e ln 2 + log m + log(1 + lo/hi) with hi = m 2^e, m in [0.5, 1):
  // |log m| < 0.7, so the single-precision log is accurate to ~1e-7 absolute
  int e2 = 0;
  const float mant = frexpf(acc.x, &e2);
  const double corr = (acc.x > 0.f && acc.x < INFINITY) ? (double)(acc.y / acc.x) : 0.0;
  const double lse = (double)M + ((double)e2 * kLn2 + (double)logf(mant) + corr);
  int st = 0;
  if (M == INFINITY || !(s == s) || s == INFINITY) st |= BASTION_STATUS_NONFINITE;
  if (M == -INFINITY) st |= BASTION_STATUS_EMPTY_ROW;
  if (st) atomicOr(&a.status[row / a.b], st);
  a.lse[row] = lse;
  return lse;
}

// --------------------------------------------------------------------------- kernels
template <int ES, int NV>
__global__ void __launch_bounds__(kT, 5) topk_cluster_kernel(TopkArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem);      // the slice's bulk copy
  uint64_t *tab_bar = bar + 1;                              // the table's arrival
  uint64_t *row_bar = bar + 2;                              // leader: the row's keys' arrival
  Scratch &sc = *reinterpret_cast<Scratch *>(smem + 128);
  // the row's thread-max prefixes [CS * 256], one copy in every CTA (the
  // leader's ranks later)
  uint16_t *keys = reinterpret_cast<uint16_t *>(smem + 128 + kScratchBytes);
  uint64_t *loc = reinterpret_cast<uint64_t *>(smem + 128 + kScratchBytes + a.tab_bytes);  // [seg]
  uint64_t *rlist = loc + a.seg;  // leader: [CS][seg], each CTA's keys, zero-padded
  // the slice (the leader's row list once its own pass is done)
  unsigned char *body = reinterpret_cast<unsigned char *>(rlist + (size_t)a.CS * a.seg);

  constexpr int NE = 16 / ES;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t rank = cluster_rank();
  const int row = blockIdx.x / a.CS;
  const int req = row / a.b;
  const Slice s = slice_at<ES>(a, row, (int)rank);

  sc.hist1[tid] = 0u;
  if (tid == 0) {
    mbar_init(bar, 1);
    mbar_init(tab_bar, 1);
    mbar_init(row_bar, 1);
    fence_mbar_init();
    sc.n_loc = 0u;
  }
  griddep_wait();
  griddep_launch_dependents();
  __syncthreads();
  if (tid == 0) {
    if (s.body) {
      mbar_arrive_expect_tx(bar, (uint32_t)s.body);
      bulk_g2s(body, reinterpret_cast<const void *>(s.ga0), (uint32_t)s.body, bar);
    }
    mbar_arrive_expect_tx(tab_bar, (uint32_t)a.CS * kT * 2);  // every CTA's prefixes
    if (rank == 0)  // every CTA's keys and share
      mbar_arrive_expect_tx(row_bar, (uint32_t)a.CS * ((uint32_t)a.seg * 8u + 16u));
  }
  cluster_arrive_relaxed();  // this CTA runs and its barriers are set
  // the unaligned head and tail of the slice (at most 2 * (NE - 1) elements):
  // one per thread, read while the copy is in flight
  const int nscal = s.nh + (s.n - s.t0);
  const bool has_x = tid < nscal;
  float xs = -INFINITY;
  uint32_t xtok = 0;
  if (has_x) {
    const int e = tid < s.nh ? tid : s.t0 + (tid - s.nh);
    xs = load_elem<ES>(s.g0 + (size_t)e * ES);
    xtok = (uint32_t)(s.e0 + e);
  }
  // one thread waits for the copy; the barrier releases the rest
  bool body_ok = true;
  if (tid == 0 && s.body) {
    body_ok = mbar_wait_bounded(bar, 0);
    if (!body_ok) atomicOr(&a.status[req], BASTION_STATUS_TIMEOUT);
  }
  __syncthreads();

  // ---- pass A: vector maxima and the thread max into the leader's table
  float vm[NV];
  float tmax = xs;
#pragma unroll
  for (int u = 0; u < NV; ++u) {
    const int v = tid + u * kT;
    vm[u] = v < s.nvec ? vmax<ES>(ld_shared_v4(body + v * 16)) : -INFINITY;
    tmax = fmaxf(tmax, vm[u]);
  }
  {
    const float wm = warp_max_f(tmax);
    if (lane == 0) sc.red_f[warp] = wm;
  }
  cluster_wait();
  {
    // this warp's 32 prefixes as four 16-byte chunks; lane k sends chunk k % 4
    // to CTA k / 4 (asynchronous stores counted on the receiver's barrier)
    const uint32_t k16 = ord_f32(tmax) >> 16;
    const int chunk = lane & 3;
    uint32_t wv[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      wv[q] = __shfl_sync(kFull, k16, chunk * 8 + 2 * q) |
              (__shfl_sync(kFull, k16, chunk * 8 + 2 * q + 1) << 16);
    const uint32_t off = (uint32_t)((rank * kT + warp * 32 + chunk * 8) * 2);
    for (int k = lane; k < 4 * a.CS; k += 32) {
      const uint32_t dst = (uint32_t)(k >> 2);
      st_async_v4(dsmem_addr(keys, dst) + off, wv[0], wv[1], wv[2], wv[3], dsmem_addr(tab_bar, dst));
    }
  }
  // sum of exp(l - m_t) while the other CTAs' prefixes arrive
  float sum = 0.f;
  if (tmax != -INFINITY) {
    // c = the float nearest tmax log2(e); every term below is off by the
    // factor 2^(tmax log2(e) - c), taken out of the sum at the end
    const float c = tmax * kL2e;
    const float c_err = fmaf(tmax, kL2e, -c);
#pragma unroll
    for (int u = 0; u < NV; ++u) {
      const int v = tid + u * kT;
      if (v < s.nvec) sum += vexp_sum<ES>(ld_shared_v4(body + v * 16), -c);
    }
    sum *= ex2(-c_err);
    if (has_x) sum += exp_shifted(xs - tmax);
  }
  const bool tab_ok = mbar_wait_bounded(tab_bar, 0);
  if (!tab_ok && lane == 0) atomicOr(&a.status[req], BASTION_STATUS_TIMEOUT);

  // ---- the row threshold: the K-th largest prefix of the table, counted by
  // its distance below the largest one (256 bins: 0..254 steps, then "more")
  const int nw = a.CS * (kT / 2);  // 32-bit words of the table, two prefixes each
  uint32_t w[kMaxCS / 2];
  uint32_t m16 = 0;
  {
    const uint32_t *tab = reinterpret_cast<const uint32_t *>(keys);
#pragma unroll
    for (int j = 0; j < kMaxCS / 2; ++j)
      if (tid + j * kT < nw) w[j] = tab[tid + j * kT];
#pragma unroll
    for (int j = 0; j < kMaxCS / 2; ++j)
      if (tid + j * kT < nw) m16 = max(m16, max(w[j] & 0xffffu, w[j] >> 16));
  }
  m16 = __reduce_max_sync(kFull, m16);
  if (lane == 0) sc.red_u[warp] = m16;
  float Mc = -INFINITY;
#pragma unroll
  for (int q = 0; q < kT / 32; ++q) Mc = fmaxf(Mc, sc.red_f[q]);
  {
    const float st = tmax == -INFINITY ? 0.f : sum * exp_shifted(tmax - Mc);
    const float2 ws = ff_warp_sum(make_float2(st, 0.f));
    if (lane == 0) sc.red_s[warp] = ws;
  }
  __syncthreads();
  uint32_t M16 = 0;
#pragma unroll
  for (int q = 0; q < kT / 32; ++q) M16 = max(M16, sc.red_u[q]);
  {
    uint32_t more = 0;
#pragma unroll
    for (int j = 0; j < kMaxCS / 2; ++j) {
      if (tid + j * kT < nw) {
        const uint32_t d0 = M16 - (w[j] & 0xffffu), d1 = M16 - (w[j] >> 16);
        if (d0 < 255u) atomicAdd(&sc.hist1[255u - d0], 1u); else ++more;
        if (d1 < 255u) atomicAdd(&sc.hist1[255u - d1], 1u); else ++more;
      }
    }
    more = __reduce_add_sync(kFull, more);
    if (lane == 0 && more) atomicAdd(&sc.hist1[0], more);
  }
  __syncthreads();
  if (warp == 0) find_digit(sc.hist1, (uint32_t)a.K, sc.digit_info, lane);
  __syncthreads();
  // a K-th prefix 255 or more steps below the largest: every element survives
  // (and the leader falls back to the exact selection if they do not fit)
  const uint32_t dK = 255u - sc.digit_info[0];
  float T = dK < 255u ? unord_f32((M16 - dK) << 16) : -INFINITY;
  if (!(T == T)) T = -INFINITY;  // the prefix of -inf maps to a NaN pattern

  // ---- pass B: this thread's elements >= T into the CTA's list
  uint32_t hmask = 0, cnt = 0;
#pragma unroll
  for (int u = 0; u < NV; ++u) hmask |= (tid + u * kT < s.nvec && vm[u] >= T ? 1u : 0u) << u;
  const bool hx = has_x && xs >= T;
  for (uint32_t hm = hmask; hm; hm &= hm - 1u) {
    float f[NE];
    unpack<ES>(ld_shared_v4(body + (tid + (__ffs(hm) - 1) * kT) * 16), f);
#pragma unroll
    for (int i = 0; i < NE; ++i) cnt += f[i] >= T ? 1u : 0u;
  }
  cnt += hx ? 1u : 0u;
  if (cnt) {
    uint32_t idx = atomicAdd(&sc.n_loc, cnt);
    const uint32_t seg = (uint32_t)a.seg;
    if (hx) {
      if (idx < seg) loc[idx] = make_key(xs, xtok);
      ++idx;
    }
    for (uint32_t hm = hmask; hm; hm &= hm - 1u) {
      const int v = tid + (__ffs(hm) - 1) * kT;
      float f[NE];
      unpack<ES>(ld_shared_v4(body + v * 16), f);
      const uint32_t tok0 = (uint32_t)(s.e0 + s.nh + v * NE);
#pragma unroll
      for (int i = 0; i < NE; ++i) {
        if (f[i] >= T) {
          if (idx < seg) loc[idx] = make_key(f[i], tok0 + (uint32_t)i);
          ++idx;
        }
      }
    }
  }
  __syncthreads();
  if (warp == 0) {
    // the CTA's keys (zero-padded to seg) and its share, by asynchronous
    // stores into the leader, counted on the leader's row barrier
    float2 acc = lane < kT / 32 ? sc.red_s[lane] : make_float2(0.f, 0.f);
    acc = ff_warp_sum(acc);
    const uint32_t nl = sc.n_loc, seg = (uint32_t)a.seg;
    const uint32_t rl = dsmem_addr(rlist, 0) + rank * seg * 8u, rb = dsmem_addr(row_bar, 0);
    for (uint32_t c = lane; c < seg / 2; c += 32) {
      const uint64_t k0 = 2 * c < nl ? loc[2 * c] : 0ull, k1 = 2 * c + 1 < nl ? loc[2 * c + 1] : 0ull;
      st_async_v4(rl + c * 16u, (uint32_t)k0, (uint32_t)(k0 >> 32), (uint32_t)k1,
                  (uint32_t)(k1 >> 32), rb);
    }
    if (lane == 0)
      st_async_v4(dsmem_addr(&sc.part[rank], 0), __float_as_uint(Mc), __float_as_uint(acc.x),
                  __float_as_uint(acc.y), nl, rb);
  }
  if (rank != 0) {
    // Nothing reads or writes a non-leader's shared memory now, unless a wait
    // above ran out: then its own bulk copy or another CTA's prefixes may
    // still be landing, and the CTA waits for them (bounded) before it leaves.
    if (!tab_ok) mbar_wait_bounded(tab_bar, 0);
    if (!body_ok) mbar_wait_bounded(bar, 0);
    return;
  }

  // ---- leader: the row's keys, their ranks, and lse (last warp) meanwhile
  const bool row_ok = mbar_wait_bounded(row_bar, 0);
  if (!row_ok && lane == 0) atomicOr(&a.status[req], BASTION_STATUS_TIMEOUT);
  uint64_t *list = reinterpret_cast<uint64_t *>(body);  // this CTA's slice is spent
  if (tid == 0) {
    int o = 0, over = 0;
    for (int r = 0; r < a.CS; ++r) {
      sc.off[r] = o;
      o += (int)min(sc.part[r].n, (uint32_t)a.seg);
      over |= sc.part[r].n > (uint32_t)a.seg;
    }
    sc.off[a.CS] = over ? -1 : o;
  }
  if (tid == kT - 32) sc.lse = row_lse(a, row, sc.part, a.CS);
  __syncthreads();
  int n = sc.off[a.CS];
  if (n >= a.K) {
    for (int i = tid; i < a.CS * a.seg; i += kT) {
      const int r = i / a.seg, j = i - r * a.seg;
      if (j < sc.off[r + 1] - sc.off[r]) list[sc.off[r] + j] = rlist[i];
    }
  } else {  // a list overflowed (or too few keys): exact selection
    const unsigned char *g = a.logits + (size_t)row * (size_t)a.ld * ES;
    n = row_topk_exact<ES>(g, a.V, a.K, list, sc);
  }
  if (tid == 0 && (n & 1)) list[n] = 0ull;
  __syncthreads();
  int *rk = reinterpret_cast<int *>(keys);  // the table is no longer read
  rank_keys(a, row, list, n, rk);
  __syncthreads();
  write_logq(a, row, list, n, rk, sc.lse);
  // after a wait that ran out, stores or copies into this CTA may still be in
  // flight: wait for them (bounded) before leaving
  if (!row_ok) mbar_wait_bounded(row_bar, 0);
  if (!tab_ok) mbar_wait_bounded(tab_bar, 0);
  if (!body_ok) mbar_wait_bounded(bar, 0);
}

// Rows too wide for the cluster path: one CTA per row, exact selection over
// global memory.
template <int ES>
__global__ void __launch_bounds__(kT) topk_exact_kernel(TopkArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  Scratch &sc = *reinterpret_cast<Scratch *>(smem + 128);
  uint64_t *list = reinterpret_cast<uint64_t *>(smem + 128 + kScratchBytes);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int row = blockIdx.x;
  const unsigned char *g = a.logits + (size_t)row * (size_t)a.ld * ES;
  griddep_wait();
  griddep_launch_dependents();
  float m = -INFINITY;
  for (int e = tid; e < a.V; e += kT) m = fmaxf(m, load_elem<ES>(g + (size_t)e * ES));
  m = warp_max_f(m);
  if (lane == 0) sc.red_f[warp] = m;
  __syncthreads();
  float M = -INFINITY;
  for (int w = 0; w < kT / 32; ++w) M = fmaxf(M, sc.red_f[w]);
  float2 sum = make_float2(0.f, 0.f);  // long per-thread runs: compensated
  if (M != -INFINITY)
    for (int e = tid; e < a.V; e += kT) {
      const float2 t = two_sum(sum.x, exp_shifted(load_elem<ES>(g + (size_t)e * ES) - M));
      sum = make_float2(t.x, sum.y + t.y);
    }
  const float2 ws = ff_warp_sum(sum);
  if (lane == 0) sc.red_s[warp] = ws;
  __syncthreads();
  if (tid == 0) {
    float2 acc = make_float2(0.f, 0.f);
    for (int w = 0; w < kT / 32; ++w) acc = ff_add(acc, sc.red_s[w]);
    sc.part[0] = Part{M, acc.x, acc.y, 0u};
    sc.lse = row_lse(a, row, sc.part, 1);
  }
  const int n = row_topk_exact<ES>(g, a.V, a.K, list, sc);
  if (tid == 0 && (n & 1)) list[n] = 0ull;
  __syncthreads();
  int *rk = reinterpret_cast<int *>(list + 2 * a.K + 2);
  rank_keys(a, row, list, n, rk);
  __syncthreads();
  write_logq(a, row, list, n, rk, sc.lse);
}


// --------------------------------------------------------------------------- stream path
// Many rows (at least two per SM): one CTA per row, all resident at once.  The
// row streams through a ring of kRing shared-memory stages filled by bulk
// copies (with an L2 evict-first policy: the row is read once); the warp that
// frees a stage last refills it.  Per stage a thread
// reads its kSV vectors into registers, frees the stage, and then
//  * keeps the stage's max (a 16-bit order-key prefix) in shared memory;
//  * adds 2^(l log2(e) - c) over its elements, where c is an integer kept at
//    floor(m log2(e)) of its running max m: when m grows, the running sum is
//    rescaled by the exact power of two 2^(c_old - c_new), so every exponent
//    stays below ~1 and the sum is exact up to the terms' own rounding.
// At the end the threads' sums are scaled to the CTA's largest c (exact
// powers of two again) and summed in two-float arithmetic: lse = c ln 2 +
// log(sum), corrected for log2(e) having been rounded to float.  T, the
// K-th largest thread max (prefix), leaves at least K elements >= T (each of
// the K largest thread maxima is one).  The (stage, thread) pairs whose max
// reaches T are listed and read again from global memory, one pair per
// thread, so that a single round of loads (microseconds while the other rows
// stream) covers them all; their elements >= T form the row's list, ranked by
// counting.  A list longer than the spent ring holds (long runs of equal
// values) hands the row to the exact selection over global memory.
constexpr int kSV = 4;                         // vectors per thread per stage
constexpr int kRing = 2;                       // stages in flight
constexpr int kStageBytes = kT * kSV * 16;     // 16 KB
constexpr float kCNone = -1.0e30f;             // c before the first finite element
constexpr int kListCap = 2048;                 // the row list's keys (the spent ring)
constexpr int kHitCap = 1024;                  // stages to read again, after the list
static_assert((kListCap + 2) * 8 + kListCap * 4 + kHitCap * 4 <= kRing * kStageBytes, "ring reuse");

// Max over a thread's kSV vectors of a stage: one chain of packed maxima.
template <int ES>
__device__ __forceinline__ float stage_max(const uint4 (&x)[kSV]) {
  if constexpr (ES == 2) {
    uint32_t m = x[0].x;
#pragma unroll
    for (int u = 0; u < kSV; ++u) {
      if (u) asm("max.bf16x2 %0, %0, %1;" : "+r"(m) : "r"(x[u].x));
      asm("max.bf16x2 %0, %0, %1;" : "+r"(m) : "r"(x[u].y));
      asm("max.bf16x2 %0, %0, %1;" : "+r"(m) : "r"(x[u].z));
      asm("max.bf16x2 %0, %0, %1;" : "+r"(m) : "r"(x[u].w));
    }
    return fmaxf(bf16lo(m), bf16hi(m));
  } else {
    float m = vmax<ES>(x[0]);
#pragma unroll
    for (int u = 1; u < kSV; ++u) m = fmaxf(m, vmax<ES>(x[u]));
    return m;
  }
}

// Sum of 2^(x log2(e) + nc) over a thread's kSV vectors of a stage: packed
// FMAs and adds, four partial sums.
template <int ES>
__device__ __forceinline__ float stage_exp_sum(const uint4 (&x)[kSV], float nc) {
  float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
  for (int u = 0; u < kSV; ++u) {
    float f[16 / ES];
    unpack<ES>(x[u], f);
#pragma unroll
    for (int i = 0; i < 16 / ES; i += 4) {
      float t0, t1, t2, t3;
      asm("{\n .reg .b64 d, e, k, c;\n"
          " mov.b64 d, {%4, %5};\n mov.b64 e, {%6, %7};\n mov.b64 k, {%9, %9};\n"
          " mov.b64 c, {%8, %8};\n fma.rn.f32x2 d, d, k, c;\n fma.rn.f32x2 e, e, k, c;\n"
          " mov.b64 {%0, %1}, d;\n mov.b64 {%2, %3}, e;\n}\n"
          : "=f"(t0), "=f"(t1), "=f"(t2), "=f"(t3)
          : "f"(f[i]), "f"(f[i + 1]), "f"(f[i + 2]), "f"(f[i + 3]), "f"(nc), "f"(kL2e));
      const float e0 = ex2(t0), e1 = ex2(t1), e2 = ex2(t2), e3 = ex2(t3);
      asm("{\n .reg .b64 a, b, p, q;\n mov.b64 a, {%0, %1};\n mov.b64 b, {%2, %3};\n"
          " mov.b64 p, {%4, %5};\n mov.b64 q, {%6, %7};\n"
          " add.rn.f32x2 a, a, p;\n add.rn.f32x2 b, b, q;\n"
          " mov.b64 {%0, %1}, a;\n mov.b64 {%2, %3}, b;\n}\n"
          : "+f"(s0), "+f"(s1), "+f"(s2), "+f"(s3)
          : "f"(e0), "f"(e1), "f"(e2), "f"(e3));
    }
  }
  return (s0 + s1) + (s2 + s3);
}


// 2^d for an integer-valued d <= 0 (0 below the normal range).
__device__ __forceinline__ float pow2_int(float d) {
  return d < -126.f ? 0.f : __int_as_float(((int)d + 127) << 23);
}

// Shared-memory layout of the stream kernel for rows of nst stages.
struct StreamLayout {
  int tkey, smax, ring, bytes;
};
__host__ __device__ inline StreamLayout stream_layout(int nst) {
  StreamLayout l;
  l.tkey = 128 + kScratchBytes;
  l.smax = l.tkey + kT * 2;
  l.ring = (l.smax + nst * kT * 2 + 127) / 128 * 128;
  l.bytes = l.ring + kRing * kStageBytes;
  return l;
}

// The K-th largest of the kT 16-bit keys at keys (16-byte aligned), two bits
// a round: the largest p with #{keys >= p} >= K.  Every lane of the calling
// warp gets it.
__device__ __forceinline__ uint32_t kth_largest_key16(const uint16_t *keys, uint32_t K, int lane) {
  const uint4 kw = ld_shared_v4(keys + lane * 8);
  const uint32_t k8[8] = {kw.x & 0xffffu, kw.x >> 16, kw.y & 0xffffu, kw.y >> 16,
                          kw.z & 0xffffu, kw.z >> 16, kw.w & 0xffffu, kw.w >> 16};
  uint32_t p = 0;
#pragma unroll 1
  for (int bit = 14; bit >= 0; bit -= 2) {
    const uint32_t c1 = p | (1u << bit), c2 = p | (2u << bit), c3 = p | (3u << bit);
    uint32_t n1 = 0, n2 = 0, n3 = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      n1 += k8[q] >= c1 ? 1u : 0u;
      n2 += k8[q] >= c2 ? 1u : 0u;
      n3 += k8[q] >= c3 ? 1u : 0u;
    }
    n1 = __reduce_add_sync(kFull, n1);
    n2 = __reduce_add_sync(kFull, n2);
    n3 = __reduce_add_sync(kFull, n3);
    p = n3 >= K ? c3 : n2 >= K ? c2 : n1 >= K ? c1 : p;
  }
  return p;
}

// The smallest float whose order-key prefix is p (-inf for the prefix of -inf).
__device__ __forceinline__ float prefix_floor(uint32_t p) {
  const float T = unord_f32(p << 16);
  return T == T ? T : -INFINITY;
}

// Elements >= T of the vectors tid + u kT (u < kSV, below lim) of stage q,
// appended to the list (count n, capacity cap).
template <int ES>
__device__ __forceinline__ void append_stage(const uint4 (&x)[kSV], int q, int lim, int tid, int nh,
                                             float T, uint64_t *list, uint32_t *n, int cap) {
  constexpr int NE = 16 / ES;
#pragma unroll
  for (int u = 0; u < kSV; ++u) {
    const int v = tid + u * kT;
    if (v >= lim) continue;
    float f[NE];
    unpack<ES>(x[u], f);
    const uint32_t tok0 = (uint32_t)(nh + (q * kStageBytes + v * 16) / ES);
#pragma unroll
    for (int i = 0; i < NE; ++i)
      if (f[i] >= T) {
        const uint32_t j = atomicAdd(n, 1u);
        if (j < (uint32_t)cap) list[j] = make_key(f[i], tok0 + (uint32_t)i);
      }
  }
}

template <int ES>
__global__ void __launch_bounds__(kT, 4) topk_stream_kernel(TopkArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t *full = reinterpret_cast<uint64_t *>(smem);            // [kRing] stage landed
  uint32_t *freed = reinterpret_cast<uint32_t *>(smem + 64);      // [kRing] warp releases
  Scratch &sc = *reinterpret_cast<Scratch *>(smem + 128);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int row = blockIdx.x;
  const int req = row / a.b;
  const Slice s = slice_at<ES>(a, row, 0);
  const int nst = (s.body + kStageBytes - 1) / kStageBytes;
  const StreamLayout L = stream_layout(a.nst);  // the row's stages, at most a.nst
  uint16_t *tkey = reinterpret_cast<uint16_t *>(smem + L.tkey);    // [kT] thread maxima
  uint16_t *smax = reinterpret_cast<uint16_t *>(smem + L.smax);    // [nst][kT] stage maxima
  unsigned char *ring = smem + L.ring;  // [kRing][kStageBytes]; later the row list
  const unsigned char *gbody = reinterpret_cast<const unsigned char *>(s.ga0);
  // the row is read once: its lines leave L2 first (37.9 against 38.3 us back to back)
  const uint64_t pol = l2_evict_first_policy();

  if (tid == 0) {
    for (int i = 0; i < kRing; ++i) {
      mbar_init(&full[i], 1);
      freed[i] = 0u;
    }
    fence_mbar_init();
    sc.n_loc = 0u;
    sc.n_hit = 0u;
  }
  griddep_wait();
  griddep_launch_dependents();
  __syncthreads();
  if (tid == 0)
    for (int st = 0; st < nst && st < kRing; ++st) {
      const uint32_t bytes = (uint32_t)min(kStageBytes, s.body - st * kStageBytes);
      mbar_arrive_expect_tx(&full[st], bytes);
      bulk_g2s_hint(ring + st * kStageBytes, gbody + (size_t)st * kStageBytes, bytes, &full[st], pol);
    }
  // the unaligned head and tail of the row, one element per thread
  const int nscal = s.nh + (s.n - s.t0);
  const bool has_x = tid < nscal;
  float xs = -INFINITY;
  uint32_t xtok = 0;
  if (has_x) {
    const int e = tid < s.nh ? tid : s.t0 + (tid - s.nh);
    xs = load_elem<ES>(s.g0 + (size_t)e * ES);
    xtok = (uint32_t)e;
  }
  float m = xs;
  float c = (xs > -INFINITY && xs < INFINITY) ? floorf(xs * kL2e) : kCNone;
  float hi = has_x ? ex2(fmaf(xs, kL2e, -c)) : 0.f, lo = 0.f;

  bool ok = true;
  for (int st = 0; st < nst; ++st) {
    const int slot = st % kRing;
    // after a wait that ran out, the thread goes on without data and waits
    // no more (every thread still reaches each barrier below)
    ok = ok && mbar_wait_bounded(&full[slot], (uint32_t)(st / kRing) & 1u);
    const unsigned char *buf = ring + slot * kStageBytes;
    const int lim = ok ? min(kStageBytes, s.body - st * kStageBytes) / 16 : 0;
    uint4 x[kSV];
#pragma unroll
    for (int u = 0; u < kSV; ++u) {
      const int v = tid + u * kT;
      x[u] = v < lim ? ld_shared_v4(buf + v * 16)
                     : (ES == 2 ? make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u)
                                : make_uint4(0xff800000u, 0xff800000u, 0xff800000u, 0xff800000u));
    }
    // the stage is free once every warp holds its vectors; the last warp
    // to let go refills it with stage st + kRing
    __syncwarp();
    if (lane == 0 && ok) {
      __threadfence_block();
      // the count only grows: every eighth arrival is a stage's last
      if (((atomicAdd(&freed[slot], 1u) + 1u) & (kT / 32 - 1)) == 0u) {
        __threadfence_block();
        const int nx = st + kRing;
        if (nx < nst) {
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          const uint32_t bytes = (uint32_t)min(kStageBytes, s.body - nx * kStageBytes);
          mbar_arrive_expect_tx(&full[slot], bytes);
          bulk_g2s_hint(ring + slot * kStageBytes, gbody + (size_t)nx * kStageBytes, bytes, &full[slot], pol);
        }
      }
    }
    const float smx = stage_max<ES>(x);
    smax[st * kT + tid] = (uint16_t)(ord_f32(smx) >> 16);
    m = fmaxf(m, smx);
    const float cn = floorf(m * kL2e);
    if (cn > c) {  // exact rescale of the running sum by 2^(c - cn)
      const float f = pow2_int(c - cn);
      hi *= f;
      lo *= f;
      c = cn;
    }
    const float ssum = stage_exp_sum<ES>(x, -c);
    const float2 t = two_sum(hi, ssum);
    hi = t.x;
    lo += t.y;
  }
  if (!ok) {
    atomicOr(&a.status[req], BASTION_STATUS_TIMEOUT);
    // let the copies that may still be in flight into this CTA end
    if (tid == 0)
      for (int j = 0; j < kRing; ++j) {
        const int q = nst - kRing + j;
        if (q >= 0) mbar_wait_bounded(&full[q % kRing], (uint32_t)(q / kRing) & 1u);
      }
  }

  // ---- the row's max, c and sum; T
  tkey[tid] = (uint16_t)(ord_f32(m) >> 16);
  {
    const float wm = warp_max_f(m), wc = warp_max_f(c);
    if (lane == 0) {
      sc.red_f[warp] = wm;
      sc.red_u[warp] = __float_as_uint(wc);
    }
  }
  __syncthreads();
  float M = -INFINITY, cM = kCNone;
#pragma unroll
  for (int q = 0; q < kT / 32; ++q) {
    M = fmaxf(M, sc.red_f[q]);
    cM = fmaxf(cM, __uint_as_float(sc.red_u[q]));
  }
  {
    const float f = c > kCNone ? pow2_int(c - cM) : 0.f;
    const float2 ws = ff_warp_sum(make_float2(hi * f, lo * f));
    if (lane == 0) sc.red_s[warp] = ws;
  }
  const uint32_t T16 = kth_largest_key16(tkey, (uint32_t)a.K, lane);
  const float T = prefix_floor(T16);

  // ---- the row list: elements >= T of the stages whose max reaches T.  The
  // (stage, thread) pairs of those stages go to a list first, so that one
  // round of loads, a pair per thread, reads them all again.
  uint64_t *list = reinterpret_cast<uint64_t *>(ring);  // the ring is spent
  uint32_t *hits = reinterpret_cast<uint32_t *>(ring + kRing * kStageBytes - 4 * kHitCap);
  if (has_x && xs >= T) {
    const uint32_t i = atomicAdd(&sc.n_loc, 1u);
    if (i < (uint32_t)kListCap) list[i] = make_key(xs, xtok);
  }
  for (int q = 0; q < nst; ++q)
    if ((uint32_t)smax[q * kT + tid] >= T16) {
      const uint32_t h = atomicAdd(&sc.n_hit, 1u);
      if (h < (uint32_t)kHitCap) hits[h] = (uint32_t)(q * kT + tid);
    }
  __syncthreads();
  const int nhit = (int)min(sc.n_hit, (uint32_t)kHitCap + 1u);
  if (nhit <= kHitCap)
    for (int h = tid; h < nhit; h += kT) {
      const int q = (int)(hits[h] / kT), t = (int)(hits[h] % kT);
      const int lim = min(kStageBytes, s.body - q * kStageBytes) / 16;
      uint4 x[kSV];
#pragma unroll
      for (int u = 0; u < kSV; ++u) {
        const int v = t + u * kT;
        if (v < lim) x[u] = ld_stream_v4(gbody + (size_t)q * kStageBytes + (size_t)v * 16);
      }
      append_stage<ES>(x, q, lim, t, s.nh, T, list, &sc.n_loc, kListCap);
    }
  __syncthreads();
  int n = (int)sc.n_loc;
  if (tid == kT - 32) {
    float2 acc = make_float2(0.f, 0.f);
    for (int q = 0; q < kT / 32; ++q) acc = ff_add(acc, sc.red_s[q]);
    int e2 = 0;
    const float mant = frexpf(acc.x, &e2);
    const double corr = (acc.x > 0.f && acc.x < INFINITY) ? (double)(acc.y / acc.x) : 0.0;
    // acc = sum_i 2^(l_i kL2e - cM) with log2(e) = kL2e + kL2eLo; the terms
    // that matter have l_i within a few units of M
    const double lse = (double)cM * kLn2 + ((double)e2 * kLn2 + (double)logf(mant) + corr) +
                       (double)M * (double)kL2eLo * kLn2;
    int stt = 0;
    const double sd = (double)acc.x + (double)acc.y;
    if (M == INFINITY || !(sd == sd) || sd == INFINITY || !(cM < INFINITY)) stt |= BASTION_STATUS_NONFINITE;
    if (M == -INFINITY) stt |= BASTION_STATUS_EMPTY_ROW;
    if (stt) atomicOr(&a.status[req], stt);
    a.lse[row] = lse;
    sc.lse = lse;
  }
  const int want = min(a.K, a.V);
  if (n < want || n > kListCap || nhit > kHitCap) {  // too few keys (non-finite rows) or too many: exact selection
    __syncthreads();
    const unsigned char *g = a.logits + (size_t)row * (size_t)a.ld * ES;
    n = row_topk_exact<ES>(g, a.V, a.K, list, sc);
  }
  if (tid == 0 && (n & 1)) list[n] = 0ull;
  __syncthreads();
  int *rk = reinterpret_cast<int *>(list + kListCap + 2);
  rank_keys(a, row, list, n, rk);
  __syncthreads();
  write_logq(a, row, list, n, rk, sc.lse);
}

struct TopkPlan {
  int CS, SL, NV, seg, tab_bytes, body_bytes, nst;
  size_t smem;
  bool exact, stream;
};

// Which kernel takes the rows: BASTION_TOPK_PATH=stream|cluster forces one
// (where it applies), otherwise the stream kernel once there are two rows
// per SM and four of its CTAs fit on an SM.
TopkPlan plan_topk(int V, int K, int es, int rows, int sms, const void *, int64_t) {
  TopkPlan p;
  p.stream = false;
  p.nst = 0;
  {
    const int nst = (int)(((size_t)V * es + kStageBytes - 1) / kStageBytes);
    const size_t smem = nst <= 64 ? (size_t)stream_layout(nst).bytes : ~(size_t)0;
    const char *force = getenv("BASTION_TOPK_PATH");
    const bool fs = force && strcmp(force, "stream") == 0, fc = force && strcmp(force, "cluster") == 0;
    const bool fits = K <= kT && nst <= 64 && smem <= 227 * 1024;
    if (fits && !fc && (fs || (rows >= 2 * sms && smem <= 56 * 1024 - 256))) {
      p.stream = true;
      p.exact = false;
      p.CS = 1;
      p.SL = V;
      p.NV = 0;
      p.seg = 0;
      p.tab_bytes = 0;
      p.body_bytes = 0;
      p.nst = nst;
      p.smem = smem;
      return p;
    }
  }

  p.exact = K > kT;  // the row threshold uses one key per thread of a CTA at least
  const int max_vec = kT * 16;  // 16 vectors per thread at most
  int cs = (V + 8191) / 8192;
  cs = cs < 1 ? 1 : (cs > 8 ? 8 : cs);
  auto slice = [&](int c) { return (((V + c - 1) / c) + 7) & ~7; };
  p.SL = slice(cs);
  if ((size_t)p.SL * es / 16 + 1 > (size_t)max_vec) {
    cs = kMaxCS;
    p.SL = slice(cs);
  }
  p.CS = cs;
  const int nvec = (int)((size_t)p.SL * es / 16 + 1);
  const int per = (nvec + kT - 1) / kT;
  p.NV = per <= 2 ? 2 : per <= 4 ? 4 : per <= 8 ? 8 : per <= 12 ? 12 : 16;
  // keys per CTA in the leader's row list: twice the fair share, >= 32, even
  p.seg = (2 * K + cs - 1) / cs;
  p.seg = ((p.seg > 32 ? p.seg : 32) + 1) & ~1;
  const int nrow = cs * p.seg;  // the row list: its keys (and a pad) and their ranks
  // the table of thread-max prefixes, later the leader's ranks
  const int tab = cs * kT * 2 > (nrow + 2) * 4 ? cs * kT * 2 : (nrow + 2) * 4;
  p.tab_bytes = (tab + 127) & ~127;
  // the slice, later the leader's compacted row list
  const size_t body = (size_t)p.SL * es > (size_t)(nrow + 2) * 8 ? (size_t)p.SL * es : (size_t)(nrow + 2) * 8;
  p.body_bytes = (int)((body + 127) / 128 * 128);
  p.smem = 128 + kScratchBytes + (size_t)p.tab_bytes + (size_t)(p.seg + nrow) * 8 +
           (size_t)p.body_bytes;
  if (per > 16 || p.smem > 227 * 1024) p.exact = true;
  if (p.exact) {
    p.CS = 1;
    p.smem = 128 + kScratchBytes + (size_t)(2 * K + 2) * 12;
  }
  return p;
}

template <int ES>
cudaError_t launch_cluster(const TopkPlan &p, const TopkArgs &a, cudaStream_t stream) {
  void (*kern)(TopkArgs) = nullptr;
  switch (p.NV) {
    case 2: kern = topk_cluster_kernel<ES, 2>; break;
    case 4: kern = topk_cluster_kernel<ES, 4>; break;
    case 8: kern = topk_cluster_kernel<ES, 8>; break;
    case 12: kern = topk_cluster_kernel<ES, 12>; break;
    default: kern = topk_cluster_kernel<ES, 16>; break;
  }
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
  if (e == cudaSuccess && p.CS > 8)
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  return launch_cluster_pdl(kern, dim3((unsigned)(a.rows * p.CS)), dim3(kT), p.smem, stream, p.CS, a);
}

}  // namespace

// The kernels keep all their state on chip; the workspace is reserved.
size_t topk_workspace_bytes(int, int, int, int, int) { return 256; }

int topk_max_smem_ok(int, int, int) { return 1; }

namespace {

TopkArgs topk_args(const TopkPlan &p, const void *logits, int B, int b, int V, int64_t ld, int K,
                   float *topk_logq, float *topk_logit, int32_t *topk_tok, double *lse,
                   int32_t *status) {
  TopkArgs a;
  a.logits = static_cast<const unsigned char *>(logits);
  a.rows = B * b;
  a.b = b;
  a.V = V;
  a.K = K;
  a.CS = p.CS;
  a.SL = p.SL;
  a.seg = p.seg;
  a.tab_bytes = p.tab_bytes;
  a.body_bytes = p.body_bytes;
  a.nst = p.nst;
  a.ld = ld;
  a.topk_logq = topk_logq;
  a.topk_logit = topk_logit;
  a.topk_tok = topk_tok;
  a.lse = lse;
  a.status = status;
  return a;
}

int sm_count() {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms;
}

cudaError_t launch_plan(const TopkPlan &p, const TopkArgs &a, int es, int sms, cudaStream_t stream) {
  cudaError_t e;
  if (p.stream) {
    auto kern = es == 4 ? topk_stream_kernel<4> : topk_stream_kernel<2>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
    if (e == cudaSuccess) e = launch_pdl(kern, dim3((unsigned)a.rows), dim3(kT), p.smem, stream, a);
  } else if (p.exact) {
    auto kern = es == 4 ? topk_exact_kernel<4> : topk_exact_kernel<2>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
    if (e == cudaSuccess) e = launch_pdl(kern, dim3((unsigned)a.rows), dim3(kT), p.smem, stream, a);
  } else {
    e = es == 4 ? launch_cluster<4>(p, a, stream) : launch_cluster<2>(p, a, stream);
  }
  return e;
}

}  // namespace

int launch_topk(const void *logits, int dtype, int B, int b, int V, int64_t ld, int K,
                float *topk_logq, float *topk_logit, int32_t *topk_tok, double *lse,
                void *, int32_t *status, cudaStream_t stream) {
  const int es = dtype == BASTION_F32 ? 4 : 2;
  const int sms = sm_count();
  const TopkPlan p = plan_topk(V, K, es, B * b, sms, logits, ld);
  const TopkArgs a = topk_args(p, logits, B, b, V, ld, K, topk_logq, topk_logit, topk_tok, lse, status);
  const cudaError_t e = launch_plan(p, a, es, sms, stream);
  return (e == cudaSuccess && cudaGetLastError() == cudaSuccess) ? BASTION_OK : BASTION_ERR_LAUNCH;
}

}  // namespace bastion
