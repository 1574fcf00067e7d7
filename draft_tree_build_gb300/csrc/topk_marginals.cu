// Step 1 of the draft-tree path: softmax + top-K marginals over the full vocab.
//
// Bastion (gist.science/nl/paper/2605.29727), Methodologie §1: the block-
// diffusion drafter emits position-wise marginals q_k = softmax(l_k); the
// children of a depth-(k-1) tree node are the ranked tokens of q_k.
//
// Design (HBM-bound sweep, one read of every logit):
//  * a row is cut into C equal chunks of at most 32 KB; one CTA per (row,
//    chunk) stages its chunk in shared memory with one TMA bulk copy
//    (cp.async.bulk), so the chunk is read from HBM once and swept twice from
//    shared memory, while the other CTAs resident on the SM keep their copies
//    in flight;
//  * sweep 1: the max of each 16-byte vector (packed bf16x2 max), kept in
//    registers, and per-thread maxima.  The chunk max M_c comes from them, and
//    so does a prefilter threshold T0: a two-pass radix select over the 16-bit
//    prefixes of the 256 thread maxima finds the K-th largest prefix, and the
//    smallest value with that prefix is reached by at least K distinct
//    elements, so every top-K element of the chunk is >= T0;
//  * sweep 2: sum of exp(l - M_c) with packed f32x2 arithmetic and ex2, the
//    log2(e) factor split in two parts so its rounding does not bias all terms
//    alike, then a compensated (two-float) reduction across threads; vectors
//    whose max reaches T0 append their elements >= T0 (about K of them);
//  * the survivors are sorted by one warp (register bitonic network on the
//    64-bit keys value desc, token asc; counting rank beyond 256 survivors, an
//    exact radix select over the chunk if they do not fit at all);
//  * the last CTA of a row to finish (atomic arrival counter, no waiting)
//    merges the chunk partials: M = max M_c, s = sum s_c exp(M_c - M) as a
//    two-float sum, lse = M + log s in fp64; the best chunk K-th key bounds
//    the row's K-th key from below, so only list entries at or above it are
//    sorted for the row's top-K.
#include <cuda_bf16.h>

#include "common.cuh"

namespace bastion {

namespace {

constexpr int kT = 256;       // threads per CTA (8 warps)
constexpr int kPad = 32;      // bytes in front of the staged chunk
constexpr float kL2eHi = 1.4426950216293335f;     // log2(e) rounded to float
constexpr float kL2eLo = 1.925963033500011e-08f;  // log2(e) - kL2eHi

struct TopkArgs {
  const unsigned char *logits;
  int rows, b, V, K, CL, C, cap, chunk_bytes, lists_bytes;
  int64_t ld;  // elements
  float *topk_logq, *topk_logit;
  int32_t *topk_tok;
  double *lse;
  int32_t *status;
  float *part_m;
  float2 *part_s;  // (hi, lo) of the chunk's sum of exp(l - M_c)
  int32_t *part_n;
  uint64_t *part_keys;
  uint32_t *row_cnt;
};

struct Scratch {
  float lanemax[kT];  // chunk maxima during the merge
  uint32_t hist2[256];
  float red_f[8];
  float2 red_s[8];
  float2 s_row;
  uint32_t hist[256];
  unsigned long long kth;
  int n_cand;
  int n_surv;
  int last;
  uint32_t digit_info[2];
  int scan[kT + 1];
};

// --------------------------------------------------------------------------- arithmetic
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// exp(x0 - m) + exp(x1 - m), exp(x2 - m) + exp(x3 - m) as a pair, with the
// subtraction and the split log2(e) product in packed f32x2 arithmetic.
__device__ __forceinline__ void exp4(float x0, float x1, float x2, float x3, float m, float &s0,
                                     float &s1) {
  float t0, t1, t2, t3;
  asm("{\n .reg .b64 d, e, mm, hh, ll, p, q;\n"
      " mov.b64 d, {%4, %5};\n mov.b64 e, {%6, %7};\n mov.b64 mm, {%8, %8};\n"
      " mov.b64 hh, {%9, %9};\n mov.b64 ll, {%10, %10};\n"
      " sub.rn.f32x2 d, d, mm;\n sub.rn.f32x2 e, e, mm;\n"
      " mul.rn.f32x2 p, d, ll;\n mul.rn.f32x2 q, e, ll;\n"
      " fma.rn.f32x2 d, d, hh, p;\n fma.rn.f32x2 e, e, hh, q;\n"
      " mov.b64 {%0, %1}, d;\n mov.b64 {%2, %3}, e;\n}\n"
      : "=f"(t0), "=f"(t1), "=f"(t2), "=f"(t3)
      : "f"(x0), "f"(x1), "f"(x2), "f"(x3), "f"(m), "f"(kL2eHi), "f"(kL2eLo));
  const float e0 = ex2(t0), e1 = ex2(t1), e2 = ex2(t2), e3 = ex2(t3);
  asm("{\n .reg .b64 a, c;\n mov.b64 a, {%2, %3};\n mov.b64 c, {%4, %5};\n"
      " add.rn.f32x2 a, a, c;\n mov.b64 {%0, %1}, a;\n}\n"
      : "=f"(s0), "=f"(s1)
      : "f"(e0), "f"(e1), "f"(e2), "f"(e3));
}

__device__ __forceinline__ float exp_shifted(float d) { return ex2(fmaf(d, kL2eHi, d * kL2eLo)); }

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

// Descending bitonic sort of one float per lane; returns this lane's value.
__device__ __forceinline__ float warp_sort_desc(float v, int lane) {
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      float o = __shfl_xor_sync(kFull, v, j);
      bool desc = (lane & k) == 0;
      bool lower = (lane & j) == 0;
      v = (desc == lower) ? fmaxf(v, o) : fminf(v, o);
    }
  }
  return v;
}

// Descending bitonic sort of NPL*32 64-bit keys, NPL per lane (element
// e = i*32 + lane lives in v[i] of that lane).
template <int NPL>
__device__ __forceinline__ void warp_bitonic_desc(uint64_t (&v)[NPL], int lane) {
  constexpr int N = NPL * 32;
#pragma unroll
  for (int k = 2; k <= N; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      if (j >= 32) {
        const int jj = j >> 5;
#pragma unroll
        for (int i = 0; i < NPL; ++i) {
          const int ip = i ^ jj;
          if (ip > i) {
            const bool desc = ((i * 32 + lane) & k) == 0;
            const uint64_t x = v[i], y = v[ip];
            const bool sw = desc ? (x < y) : (x > y);
            v[i] = sw ? y : x;
            v[ip] = sw ? x : y;
          }
        }
      } else {
        const bool lower = (lane & j) == 0;
#pragma unroll
        for (int i = 0; i < NPL; ++i) {
          const uint64_t o = __shfl_xor_sync(kFull, v[i], j);
          const bool desc = ((i * 32 + lane) & k) == 0;
          const bool keep_max = desc == lower;
          v[i] = keep_max ? (v[i] > o ? v[i] : o) : (v[i] < o ? v[i] : o);
        }
      }
    }
  }
}

// Sort n <= NPL*32 keys from src (descending) with warp 0 and write the first
// min(n, K) of them to dst.
template <int NPL>
__device__ __forceinline__ void warp_sort_write(const uint64_t *src, int n, int K, uint64_t *dst,
                                                int lane) {
  uint64_t v[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int e = i * 32 + lane;
    v[i] = e < n ? src[e] : 0ull;
  }
  warp_bitonic_desc<NPL>(v, lane);
  const int lim = min(n, K);
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int e = i * 32 + lane;
    if (e < lim) dst[e] = v[i];
  }
}

// Rank n unique keys of src exactly and write the first min(n, K), sorted
// descending, to dst (all threads of the CTA call it; a barrier must follow
// before dst is read when dst is shared memory).
__device__ __forceinline__ void sort_top(const uint64_t *src, int n, int K, uint64_t *dst) {
  const int tid = threadIdx.x, lane = tid & 31;
  if (n <= 64) {
    if (tid < 32) warp_sort_write<2>(src, n, K, dst, lane);
  } else if (n <= 128) {
    if (tid < 32) warp_sort_write<4>(src, n, K, dst, lane);
  } else if (n <= 256) {
    if (tid < 32) warp_sort_write<8>(src, n, K, dst, lane);
  } else {
    for (int i = tid; i < n; i += kT) {
      const uint64_t ki = src[i];
      int rk = 0;
      for (int j = 0; j < n; ++j) rk += src[j] > ki;
      if (rk < K) dst[rk] = ki;
    }
  }
}

// Number of entries >= c in a descending list of 32.
__device__ __forceinline__ int count_ge(const float *list, float c) {
  int lo = 0, hi = 32;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (list[mid] >= c) lo = mid + 1; else hi = mid;
  }
  return lo;
}

// --------------------------------------------------------------------------- chunk geometry
struct Item {
  int row, c, e0, n, body, nh, t0, nvec;
  const unsigned char *g0;
  uintptr_t ga0;
};

template <int ES>
__device__ __forceinline__ Item item_at(const TopkArgs &a, int it) {
  Item m;
  m.row = it / a.C;
  m.c = it - m.row * a.C;
  m.e0 = m.c * a.CL;
  m.n = min(a.V - m.e0, a.CL);
  m.g0 = a.logits + ((size_t)m.row * (size_t)a.ld + (size_t)m.e0) * ES;
  m.ga0 = ((uintptr_t)m.g0 + 15) & ~(uintptr_t)15;
  const uintptr_t ga1 = ((uintptr_t)m.g0 + (uintptr_t)m.n * ES) & ~(uintptr_t)15;
  m.body = ga1 > m.ga0 ? (int)(ga1 - m.ga0) : 0;
  const int h = m.body ? (int)(m.ga0 - (uintptr_t)m.g0) : m.n * ES;
  m.nh = h / ES;
  m.t0 = (h + m.body) / ES;
  m.nvec = m.body / 16;
  return m;
}

// Element e of the item: from the staged body, else from global memory.
template <int ES>
__device__ __forceinline__ float item_elem(const Item &m, const unsigned char *body, int e) {
  if (e >= m.nh && e < m.t0) return load_elem<ES>(body + (size_t)(e - m.nh) * ES);
  return load_elem<ES>(m.g0 + (size_t)e * ES);
}

// Exact top-min(K, n) of the chunk when the prefilter left too many survivors:
// radix select of the K-th largest value (8-bit digits of the order-preserving
// key), then every element above it plus the lowest-token elements equal to it.
template <int ES>
__device__ void chunk_topk_exact(const Item &m, const unsigned char *body, int K, uint64_t *surv,
                                 Scratch &sc) {
  const int tid = threadIdx.x, n = m.n;
  int kk = min(K, n);
  uint32_t prefix = 0, pmask = 0;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += kT) sc.hist[i] = 0;
    __syncthreads();
    for (int e = tid; e < n; e += kT) {
      const uint32_t o = ord_f32(item_elem<ES>(m, body, e));
      if ((o & pmask) == prefix) atomicAdd(&sc.hist[(o >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (tid < 32) {
      uint32_t cnt[8], tot = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) { cnt[q] = sc.hist[255 - 8 * tid - q]; tot += cnt[q]; }
      uint32_t incl = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        uint32_t y = __shfl_up_sync(kFull, incl, o);
        if (tid >= o) incl += y;
      }
      const uint32_t above = incl - tot;
      if (above < (uint32_t)kk && incl >= (uint32_t)kk) {
        uint32_t run = above;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          if (run + cnt[q] >= (uint32_t)kk) {
            sc.digit_info[0] = 255u - 8u * tid - q;
            sc.digit_info[1] = run;
            break;
          }
          run += cnt[q];
        }
      }
    }
    __syncthreads();
    const uint32_t digit = sc.digit_info[0];
    kk -= (int)sc.digit_info[1];
    prefix |= digit << shift;
    pmask |= 255u << shift;
    __syncthreads();
  }
  if (tid == 0) sc.n_surv = 0;
  const int per = (n + kT - 1) / kT;
  const int lo = min(n, tid * per), hi = min(n, lo + per);
  int eq = 0;
  for (int e = lo; e < hi; ++e) eq += ord_f32(item_elem<ES>(m, body, e)) == prefix;
  sc.scan[tid] = eq;
  __syncthreads();
  if (tid == 0) {
    int run = 0;
    for (int t = 0; t < kT; ++t) { int v = sc.scan[t]; sc.scan[t] = run; run += v; }
  }
  __syncthreads();
  int rank_eq = sc.scan[tid];
  for (int e = lo; e < hi; ++e) {
    const float v = item_elem<ES>(m, body, e);
    const uint32_t o = ord_f32(v);
    bool take = o > prefix;
    if (o == prefix) { take = rank_eq < kk; ++rank_eq; }
    if (take) surv[atomicAdd(&sc.n_surv, 1)] = make_key(v, (uint32_t)(m.e0 + e));
  }
  __syncthreads();
}

// Append this lane's elements >= T0 of one vector (keys into surv).
template <int NE>
__device__ __forceinline__ void append_lane(const float (&f)[NE], float T0, uint32_t tok0,
                                            uint64_t *surv, int *n_surv, int cap) {
  uint32_t msk = 0;
#pragma unroll
  for (int i = 0; i < NE; ++i) msk |= (f[i] >= T0 ? 1u : 0u) << i;
  int idx = atomicAdd(n_surv, __popc(msk));
  while (msk) {
    const int i = __ffs(msk) - 1;
    msk &= msk - 1u;
    float fi = f[0];
#pragma unroll
    for (int q = 1; q < NE; ++q) fi = q == i ? f[q] : fi;
    if (idx < cap) surv[idx] = make_key(fi, tok0 + (uint32_t)i);
    ++idx;
  }
}

// Radix select of a threshold over the 16-bit prefixes of one value per
// thread: returns the smallest float whose order key has the K-th largest
// prefix (so >= K threads hold a value >= it).  All threads call it.
__device__ __forceinline__ float kth_prefix_threshold(float v, int K, Scratch &sc) {
  const int tid = threadIdx.x, lane = tid & 31;
  const uint32_t key = ord_f32(v) >> 16;
  sc.hist[tid] = 0u;
  sc.hist2[tid] = 0u;
  __syncthreads();
  atomicAdd(&sc.hist[key >> 8], 1u);
  __syncthreads();
  // digit d scanned from 255 down: lane owns digits 255-8*lane .. 255-8*lane-7
  auto find = [&](const uint32_t *h, uint32_t need) {
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
          sc.digit_info[0] = 255u - 8u * lane - q;
          sc.digit_info[1] = run;
          break;
        }
        run += cnt[q];
      }
    }
  };
  if (tid < 32) find(sc.hist, (uint32_t)K);
  __syncthreads();
  const uint32_t d1 = sc.digit_info[0], above1 = sc.digit_info[1];
  if ((key >> 8) == d1) atomicAdd(&sc.hist2[key & 255u], 1u);
  __syncthreads();
  if (tid < 32) find(sc.hist2, (uint32_t)K - above1);
  __syncthreads();
  const uint32_t t16 = (d1 << 8) | sc.digit_info[0];
  const float t = unord_f32(t16 << 16);
  return t == t ? t : -INFINITY;  // the prefix of -inf maps to a NaN pattern
}

template <int ES>
__global__ void __launch_bounds__(kT, 4) topk_kernel(TopkArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem);
  uint64_t *surv = reinterpret_cast<uint64_t *>(smem + 128);  // [cap]
  Scratch &sc = *reinterpret_cast<Scratch *>(smem + 128 + (size_t)a.cap * 8);
  uint64_t *lists = reinterpret_cast<uint64_t *>(smem + 128 + (size_t)a.cap * 8 +
                                                 ((sizeof(Scratch) + 127) / 128) * 128);
  unsigned char *chunk = reinterpret_cast<unsigned char *>(lists) + a.lists_bytes;
  unsigned char *body = chunk + kPad;

  constexpr int NE = 16 / ES;
  constexpr int kVPT = 8;  // vectors per thread (chunks hold at most 8 * 256 vectors)
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const Item m = item_at<ES>(a, blockIdx.x);
  const int req = m.row / a.b;

  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
    sc.n_surv = 0;
  }
  griddep_wait();
  griddep_launch_dependents();
  __syncthreads();
  if (tid == 0 && m.body) {
    mbar_arrive_expect_tx(bar, (uint32_t)m.body);
    bulk_g2s(body, reinterpret_cast<const void *>(m.ga0), (uint32_t)m.body, bar);
  }
  // unaligned head and tail elements: plain loads (read before the wait)
  const int nscal = m.nh + (m.n - m.t0);
  float tmax = -INFINITY;
  for (int j = tid; j < nscal; j += kT) {
    const int e = j < m.nh ? j : m.t0 + (j - m.nh);
    tmax = fmaxf(tmax, load_elem<ES>(m.g0 + (size_t)e * ES));
  }
  // one thread waits for the bulk copy; the barrier below releases the rest
  // (spinning in every thread would take issue slots from the other CTAs)
  if (tid == 0 && m.body && !mbar_wait_bounded(bar, 0)) atomicOr(&a.status[req], BASTION_STATUS_TIMEOUT);
  __syncthreads();

  // ---- sweep 1: vector maxima (kept), thread maxima, chunk max, T0
  float vm[kVPT];
#pragma unroll
  for (int u = 0; u < kVPT; ++u) {
    const int v = tid + u * kT;
    vm[u] = v < m.nvec ? vmax<ES>(ld_shared_v4(body + v * 16)) : -INFINITY;
    tmax = fmaxf(tmax, vm[u]);
  }
  {
    const float wm = warp_max_f(tmax);
    if (lane == 0) sc.red_f[warp] = wm;
  }
  float T0 = -INFINITY;
  if (a.K <= kT) T0 = kth_prefix_threshold(tmax, a.K, sc);  // has barriers
  else __syncthreads();                                     // the maxima above
  float M = -INFINITY;
#pragma unroll
  for (int w = 0; w < kT / 32; ++w) M = fmaxf(M, sc.red_f[w]);
  const bool have_mass = M != -INFINITY;

  // ---- sweep 2: sum of exp(l - M) and survivors >= T0
  float sum = 0.f;
  const uint32_t tok_vec0 = (uint32_t)(m.e0 + m.nh);
#pragma unroll
  for (int u = 0; u < kVPT; ++u) {
    const int v = tid + u * kT;
    if (v < m.nvec) {
      const uint4 x = ld_shared_v4(body + v * 16);
      float f[NE];
      unpack<ES>(x, f);
      if constexpr (ES == 2) {
        float p0, p1, q0, q1;
        exp4(f[0], f[1], f[2], f[3], M, p0, p1);
        exp4(f[4], f[5], f[6], f[7], M, q0, q1);
        sum += (p0 + p1) + (q0 + q1);
      } else {
        float p0, p1;
        exp4(f[0], f[1], f[2], f[3], M, p0, p1);
        sum += p0 + p1;
      }
      if (vm[u] >= T0) append_lane<NE>(f, T0, tok_vec0 + (uint32_t)(v * NE), surv, &sc.n_surv, a.cap);
    }
  }
  for (int j = tid; j < nscal; j += kT) {  // head and tail
    const int e = j < m.nh ? j : m.t0 + (j - m.nh);
    const float f[1] = {load_elem<ES>(m.g0 + (size_t)e * ES)};
    sum += exp_shifted(f[0] - M);
    if (f[0] >= T0) append_lane<1>(f, T0, (uint32_t)(m.e0 + e), surv, &sc.n_surv, a.cap);
  }
  {
    const float2 ws = ff_warp_sum(make_float2(sum, 0.f));
    if (lane == 0) sc.red_s[warp] = ws;
  }
  __syncthreads();  // B

  int n_s = sc.n_surv;
  if (n_s > a.cap) {
    chunk_topk_exact<ES>(m, body, a.K, surv, sc);
    n_s = sc.n_surv;
  }
  // ---- the chunk's sorted top list
  const size_t part = (size_t)m.row * a.C + m.c;
  sort_top(surv, n_s, a.K, a.part_keys + part * a.K);
  if (tid == 0) {
    float2 st = make_float2(0.f, 0.f);
    for (int w = 0; w < kT / 32; ++w) st = ff_add(st, sc.red_s[w]);
    a.part_m[part] = M;
    a.part_s[part] = have_mass ? st : make_float2(0.f, 0.f);
    a.part_n[part] = min(n_s, a.K);
  }
  __threadfence();
  __syncthreads();  // C
  if (tid == 0) sc.last = atomicAdd(&a.row_cnt[m.row], 1u) == (uint32_t)(a.C - 1);
  __syncthreads();  // D
  if (!sc.last) return;
  __threadfence();

  // ---- merge of the row's chunk partials (last arriving CTA)
  const size_t part0 = (size_t)m.row * a.C;
  float *pm = sc.lanemax;  // [C] chunk maxima (C <= 256)
  int *offs = sc.scan;     // [C + 1] list starts
  if (tid < a.C) {
    pm[tid] = __ldcg(&a.part_m[part0 + tid]);
    offs[tid + 1] = __ldcg(&a.part_n[part0 + tid]);
  }
  if (tid == 0) { sc.kth = 0ull; sc.n_cand = 0; }
  __syncthreads();
  // the best chunk K-th key: every chunk holding K keys has K keys >= its K-th
  if (tid < a.C && offs[tid + 1] == a.K) {
    const uint64_t kth = __ldcg(&a.part_keys[(part0 + tid) * a.K + a.K - 1]);
    atomicMax(reinterpret_cast<unsigned long long *>(&sc.kth), (unsigned long long)kth);
  }
  if (tid == 0) {
    offs[0] = 0;
    for (int q = 0; q < a.C; ++q) offs[q + 1] += offs[q];
  }
  float Mrow = -INFINITY;
  for (int q = 0; q < a.C; ++q) Mrow = fmaxf(Mrow, pm[q]);
  if (warp == 0) {
    float2 acc = make_float2(0.f, 0.f);
    for (int q = lane; q < a.C; q += 32) {
      const float mq = pm[q];
      if (mq != -INFINITY) {
        const float2 sq = __ldcg(&a.part_s[part0 + q]);
        const float e = expf(mq - Mrow);
        const float ph = sq.x * e;
        const float pl = fmaf(sq.x, e, -ph) + sq.y * e;
        acc = ff_add(acc, make_float2(ph, pl));
      }
    }
    acc = ff_warp_sum(acc);
    if (lane == 0) sc.s_row = acc;
  }
  __syncthreads();
  // candidates: list entries at or above the bound (at least K of them)
  const int total = offs[a.C];
  const uint64_t bound = sc.kth;
  for (int i = tid; i < total; i += kT) {
    int q = 0;
    while (offs[q + 1] <= i) ++q;
    const uint64_t key = __ldcg(&a.part_keys[(part0 + q) * a.K + (i - offs[q])]);
    if (key >= bound) lists[atomicAdd(&sc.n_cand, 1)] = key;
  }
  __syncthreads();
  sort_top(lists, sc.n_cand, a.K, surv);
  __shared__ double s_lse;
  if (tid == 0) {
    const float2 sr = sc.s_row;
    const double acc = (double)sr.x + (double)sr.y;
    const double lse = (double)Mrow + log(acc);
    s_lse = lse;
    int st = 0;
    if (Mrow == INFINITY || !(acc == acc) || acc == INFINITY) st |= BASTION_STATUS_NONFINITE;
    if (Mrow == -INFINITY) st |= BASTION_STATUS_EMPTY_ROW;
    if (st) atomicOr(&a.status[req], st);
    a.lse[m.row] = lse;
    a.row_cnt[m.row] = 0u;
  }
  __syncthreads();
  const double lse = s_lse;
  for (int j = tid; j < a.K; j += kT) {
    const uint64_t key = surv[j];
    const float v = key_value(key);
    const size_t o = (size_t)m.row * a.K + j;
    a.topk_logit[o] = v;
    a.topk_tok[o] = (int32_t)key_token(key);
    if (a.topk_logq) a.topk_logq[o] = (float)((double)v - lse);
  }
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

struct TopkPlan {
  int CL, C, cap, chunk_bytes, lists_bytes;
  size_t smem;
};

TopkPlan plan_topk(int V, int K, int es) {
  // chunks of at most 32 KB (2048 vectors of 16 bytes, 8 per thread); the
  // merge buffer holds C lists of K keys
  TopkPlan p;
  const int cl_max = es == 2 ? 16384 : 8192;
  p.C = (V + cl_max - 1) / cl_max;
  p.CL = (V + p.C - 1) / p.C;
  p.CL = (p.CL + 7) & ~7;
  p.cap = ((K > 512 ? K : 512) + 15) & ~15;  // keeps every later section 16-byte aligned
  p.chunk_bytes = (int)(((size_t)kPad + (size_t)p.CL * es + 32 + 127) / 128 * 128);
  p.lists_bytes = (int)(((size_t)p.C * K * 8 + 127) / 128 * 128);
  p.smem = 128 + (size_t)p.cap * 8 + ((sizeof(Scratch) + 127) / 128) * 128 + p.lists_bytes +
           p.chunk_bytes;
  return p;
}

}  // namespace

size_t topk_workspace_bytes(int B, int b, int V, int K, int es) {
  TopkPlan p = plan_topk(V, K, es);
  size_t R = (size_t)B * b, P = R * p.C;
  return align256(P * 4) + align256(P * 8) + align256(P * 4) + align256(P * K * 8) + align256(R * 4);
}

int topk_max_smem_ok(int V, int K, int es) {
  TopkPlan p = plan_topk(V, K, es);
  return p.C <= 256 && p.smem <= 227 * 1024;
}

int launch_topk(const void *logits, int dtype, int B, int b, int V, int64_t ld, int K,
                float *topk_logq, float *topk_logit, int32_t *topk_tok, double *lse,
                void *ws, int32_t *status, cudaStream_t stream) {
  const int es = dtype == BASTION_F32 ? 4 : 2;
  TopkPlan p = plan_topk(V, K, es);
  TopkArgs a;
  a.logits = static_cast<const unsigned char *>(logits);
  a.rows = B * b;
  a.b = b;
  a.V = V;
  a.K = K;
  a.CL = p.CL;
  a.C = p.C;
  a.cap = p.cap;
  a.chunk_bytes = p.chunk_bytes;
  a.lists_bytes = p.lists_bytes;
  a.ld = ld;
  a.topk_logq = topk_logq;
  a.topk_logit = topk_logit;
  a.topk_tok = topk_tok;
  a.lse = lse;
  a.status = status;
  size_t R = (size_t)B * b, P = R * p.C;
  unsigned char *w = static_cast<unsigned char *>(ws);
  a.part_m = reinterpret_cast<float *>(w);
  w += align256(P * 4);
  a.part_s = reinterpret_cast<float2 *>(w);
  w += align256(P * 8);
  a.part_n = reinterpret_cast<int32_t *>(w);
  w += align256(P * 4);
  a.part_keys = reinterpret_cast<uint64_t *>(w);
  w += align256(P * K * 8);
  a.row_cnt = reinterpret_cast<uint32_t *>(w);
  auto kern = es == 4 ? topk_kernel<4> : topk_kernel<2>;
  if (p.smem > 48 * 1024)
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
  const cudaError_t e = launch_pdl(kern, dim3((unsigned)P), dim3(kT), p.smem, stream, a);
  return (e == cudaSuccess && cudaGetLastError() == cudaSuccess) ? BASTION_OK : BASTION_ERR_LAUNCH;
}

}  // namespace bastion
