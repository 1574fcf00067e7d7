// Step 1 of the draft-tree path: softmax + top-K marginals over the full vocab.
//
// Bastion (gist.science/nl/paper/2605.29727), Methodologie §1: the block-
// diffusion drafter emits position-wise marginals q_k = softmax(l_k); the
// children of a depth-(k-1) tree node are the ranked tokens of q_k.
//
// Design (HBM-bound sweep, one read of every logit):
//  * a row is cut into chunks of CL elements; one CTA per (row, chunk) stages
//    its chunk in shared memory with one TMA bulk copy (cp.async.bulk), so the
//    chunk is read from HBM once and swept twice from shared memory;
//  * sweep 1: per-thread maxima.  The chunk max M_c comes from them, and so
//    does a prefilter threshold T0: in each of the 8 warps the ceil(K/8)-th
//    largest lane maximum is a value that at least ceil(K/8) distinct elements
//    of that warp reach, so the minimum over warps is reached by >= K elements
//    and every top-K element of the chunk is >= T0;
//  * sweep 2: sum of exp(l - M_c) (fp32 per 8-element vector, Kahan-compensated
//    per thread, fp64 across threads) and compaction of the few elements >= T0;
//  * the survivors are ranked exactly by counting (keys are unique: value desc,
//    token asc); if they do not fit (heavy ties at T0) an exact radix select
//    over the whole chunk takes over;
//  * the last CTA of a row to finish (atomic arrival counter, no waiting)
//    merges the chunk partials: M = max M_c, s = sum s_c exp(M_c - M) in fp64,
//    lse = M + log s, and the top-K of the union of the sorted chunk lists by
//    rank = own position + binary-search counts in the other lists.
#include <cuda_bf16.h>

#include <type_traits>

#include "common.cuh"

namespace bastion {

namespace {

constexpr int kT = 256;     // threads per CTA (8 warps)
constexpr int kCap = 1024;  // survivor keys held in shared memory (>= max K)
constexpr int kPad = 32;    // bytes in front of the staged chunk (head elements)
constexpr float kL2eHi = 1.4426950216293335f;   // log2(e) rounded to float
constexpr float kL2eLo = 1.925963033500011e-08f;  // log2(e) - kL2eHi

struct TopkArgs {
  const unsigned char *logits;
  int rows, b, V, K, CL, C;
  int64_t ld;  // elements
  float *topk_logq, *topk_logit;
  int32_t *topk_tok;
  double *lse;
  int32_t *status;
  float *part_m;
  double *part_s;
  int32_t *part_n;
  uint64_t *part_keys;
  uint32_t *row_cnt;
};

struct Scratch {
  float red_f[32];
  double red_d[32];
  uint32_t hist[256];
  int n_surv;
  int last;
  float M;
  float T0;
  uint32_t digit_info[2];
  int scan[kT + 1];
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// exp(d) for d = l - M <= 0 with the log2(e) product split in two parts, so
// the constant's rounding does not bias every term the same way.
__device__ __forceinline__ float exp_shifted(float d) {
  return ex2(fmaf(d, kL2eHi, d * kL2eLo));
}

template <int ES>
__device__ __forceinline__ float load_elem_smem(const unsigned char *p) {
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

// Append the elements of one lane that pass `pass[i]` as keys into surv[].
template <int NE>
__device__ __forceinline__ void append_keys(const float (&f)[NE], const bool (&pass)[NE],
                                            uint32_t tok0, int lane, uint64_t *surv,
                                            int *n_surv) {
#pragma unroll
  for (int i = 0; i < NE; ++i) {
    unsigned bal = __ballot_sync(kFull, pass[i]);
    if (bal) {
      int leader = __ffs(bal) - 1;
      int base = 0;
      if (lane == leader) base = atomicAdd(n_surv, __popc(bal));
      base = __shfl_sync(kFull, base, leader);
      if (pass[i]) {
        int idx = base + __popc(bal & ((1u << lane) - 1u));
        if (idx < kCap) surv[idx] = make_key(f[i], tok0 + (uint32_t)i);
      }
    }
  }
}

// Exact top-min(K, n) of the chunk when the prefilter left too many survivors:
// radix select of the K-th largest value (8-bit digits of the order-preserving
// key), then every element above it plus the lowest-token elements equal to it.
template <int ES>
__device__ void chunk_topk_exact(const unsigned char *elem0, int n, int K, uint32_t tok_base,
                                 uint64_t *surv, Scratch &sc) {
  const int tid = threadIdx.x;
  int kk = min(K, n);
  uint32_t prefix = 0, pmask = 0;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += kT) sc.hist[i] = 0;
    __syncthreads();
    for (int e = tid; e < n; e += kT) {
      uint32_t o = ord_f32(load_elem_smem<ES>(elem0 + (size_t)e * ES));
      if ((o & pmask) == prefix) atomicAdd(&sc.hist[(o >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (tid < 32) {
      // bins 255 - 8*lane ... 255 - 8*lane - 7 (descending digits)
      uint32_t cnt[8], tot = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) { cnt[q] = sc.hist[255 - 8 * tid - q]; tot += cnt[q]; }
      uint32_t incl = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        uint32_t y = __shfl_up_sync(kFull, incl, o);
        if (tid >= o) incl += y;
      }
      uint32_t above = incl - tot;  // count in higher digit bins than this lane's
      bool mine = above < (uint32_t)kk && incl >= (uint32_t)kk;
      if (mine) {
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
    uint32_t digit = sc.digit_info[0];
    kk -= (int)sc.digit_info[1];
    prefix |= digit << shift;
    pmask |= 255u << shift;
    __syncthreads();
  }
  // prefix = order key of the K-th largest value; take kk elements equal to it
  // in token order, and every element above it.
  if (tid == 0) sc.n_surv = 0;
  const int per = (n + kT - 1) / kT;
  const int lo = min(n, tid * per), hi = min(n, lo + per);
  int eq = 0;
  for (int e = lo; e < hi; ++e) eq += ord_f32(load_elem_smem<ES>(elem0 + (size_t)e * ES)) == prefix;
  sc.scan[tid] = eq;
  __syncthreads();
  if (tid == 0) {
    int run = 0;
    for (int t = 0; t < kT; ++t) { int v = sc.scan[t]; sc.scan[t] = run; run += v; }
  }
  __syncthreads();
  int rank_eq = sc.scan[tid];
  for (int e = lo; e < hi; ++e) {
    float v = load_elem_smem<ES>(elem0 + (size_t)e * ES);
    uint32_t o = ord_f32(v);
    bool take = o > prefix;
    if (o == prefix) { take = rank_eq < kk; ++rank_eq; }
    if (take) {
      int idx = atomicAdd(&sc.n_surv, 1);
      surv[idx] = make_key(v, tok_base + (uint32_t)e);
    }
  }
  __syncthreads();
}

template <int ES>
__global__ void __launch_bounds__(kT, 4) topk_chunk_kernel(TopkArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem);
  uint64_t *surv = reinterpret_cast<uint64_t *>(smem + 16);
  Scratch &sc = *reinterpret_cast<Scratch *>(smem + 16 + kCap * 8);
  unsigned char *buf = smem + 16 + kCap * 8 + ((sizeof(Scratch) + 127) / 128) * 128;

  constexpr int NE = 16 / ES;  // elements per 16-byte vector
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int row = blockIdx.x / a.C, c = blockIdx.x % a.C;
  const int req = row / a.b;
  const int e0 = c * a.CL;
  const int n = min(a.V - e0, a.CL);
  const unsigned char *g0 = a.logits + ((size_t)row * (size_t)a.ld + (size_t)e0) * ES;
  const uintptr_t ga0 = ((uintptr_t)g0 + 15) & ~(uintptr_t)15;
  const uintptr_t ga1 = ((uintptr_t)g0 + (uintptr_t)n * ES) & ~(uintptr_t)15;
  const int body = ga1 > ga0 ? (int)(ga1 - ga0) : 0;       // bytes copied in bulk
  const int h = body ? (int)(ga0 - (uintptr_t)g0) : n * ES;  // head bytes
  const int nh = h / ES;                                      // head elements
  const int t0 = (h + body) / ES;                             // first tail element
  const int nvec = body / 16;
  unsigned char *elem0 = buf + kPad - h;  // chunk element e lives at elem0 + e*ES

  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
    sc.n_surv = 0;
  }
  __syncthreads();
  if (tid == 0 && body) {
    mbar_arrive_expect_tx(bar, (uint32_t)body);
    bulk_g2s(buf + kPad, reinterpret_cast<const void *>(ga0), (uint32_t)body, bar);
  }
  // unaligned head and tail elements: plain loads
  using ElemT = typename std::conditional<ES == 4, uint32_t, uint16_t>::type;
  for (int e = tid; e < nh; e += kT)
    reinterpret_cast<ElemT *>(elem0)[e] = reinterpret_cast<const ElemT *>(g0)[e];
  for (int e = t0 + tid; e < n; e += kT)
    reinterpret_cast<ElemT *>(elem0)[e] = reinterpret_cast<const ElemT *>(g0)[e];
  if (body && !mbar_wait_bounded(bar, 0)) {
    if (lane == 0) atomicOr(&a.status[req], BASTION_STATUS_TIMEOUT);
  }
  __syncthreads();

  // ---- sweep 1: maxima
  float tmax = -INFINITY;
  for (int v = tid; v < nvec; v += kT) tmax = fmaxf(tmax, vmax<ES>(ld_shared_v4(buf + kPad + v * 16)));
  for (int e = tid; e < nh; e += kT) tmax = fmaxf(tmax, load_elem_smem<ES>(elem0 + (size_t)e * ES));
  for (int e = t0 + tid; e < n; e += kT) tmax = fmaxf(tmax, load_elem_smem<ES>(elem0 + (size_t)e * ES));
  {
    float wm = warp_max_f(tmax);
    float sorted = warp_sort_desc(tmax, lane);
    const int kw = (a.K + 7) / 8;
    float tw = __shfl_sync(kFull, sorted, kw <= 32 ? kw - 1 : 0);
    if (kw > 32) tw = -INFINITY;
    if (lane == 0) { sc.red_f[warp] = wm; sc.red_f[8 + warp] = tw; }
  }
  __syncthreads();
  if (tid == 0) {
    float m = -INFINITY, t = INFINITY;
    for (int w = 0; w < kT / 32; ++w) { m = fmaxf(m, sc.red_f[w]); t = fminf(t, sc.red_f[8 + w]); }
    sc.M = m;
    sc.T0 = t;
  }
  __syncthreads();
  const float M = sc.M, T0 = sc.T0;
  const bool have_mass = M != -INFINITY;

  // ---- sweep 2: sum of exp(l - M) and survivors >= T0
  float s = 0.f, comp = 0.f;
  const uint32_t tok_vec0 = (uint32_t)(e0 + h / ES);  // token of the first body element
  for (int base = warp * 32; base < nvec; base += kT) {
    const int v = base + lane;
    const bool valid = v < nvec;
    float f[NE];
    uint4 x = make_uint4(0, 0, 0, 0);
    if (valid) x = ld_shared_v4(buf + kPad + v * 16);
    unpack<ES>(x, f);
    float vs = 0.f;
    bool any = false;
    bool pass[NE];
#pragma unroll
    for (int i = 0; i < NE; ++i) {
      vs += exp_shifted(f[i] - M);
      pass[i] = valid && f[i] >= T0;
      any |= pass[i];
    }
    if (valid && have_mass) {
      float y = vs - comp;
      float t = s + y;
      comp = (t - s) - y;
      s = t;
    }
    if (__any_sync(kFull, any))
      append_keys<NE>(f, pass, tok_vec0 + (uint32_t)(v * NE), lane, surv, &sc.n_surv);
  }
  // head and tail scalars, by warp 0
  if (warp == 0) {
    const int nscal = nh + (n - t0);
    for (int base = 0; base < nscal; base += 32) {
      const int j = base + lane;
      const bool valid = j < nscal;
      const int e = j < nh ? j : t0 + (j - nh);
      float f[1] = {valid ? load_elem_smem<ES>(elem0 + (size_t)e * ES) : -INFINITY};
      bool pass[1] = {valid && f[0] >= T0};
      if (valid && have_mass) {
        float y = exp_shifted(f[0] - M) - comp;
        float t = s + y;
        comp = (t - s) - y;
        s = t;
      }
      if (__any_sync(kFull, pass[0]))
        append_keys<1>(f, pass, (uint32_t)(e0 + e), lane, surv, &sc.n_surv);
    }
  }
  double sd = warp_sum_d((double)s - (double)comp);
  if (lane == 0) sc.red_d[warp] = sd;
  __syncthreads();

  int n_s = sc.n_surv;
  if (n_s > kCap) {
    chunk_topk_exact<ES>(elem0, n, a.K, (uint32_t)e0, surv, sc);
    n_s = sc.n_surv;
  }
  // ---- rank survivors exactly and write the chunk's sorted top list
  const size_t part = (size_t)row * a.C + c;
  uint64_t *out_keys = a.part_keys + part * a.K;
  for (int i = tid; i < n_s; i += kT) {
    const uint64_t ki = surv[i];
    int rk = 0;
    for (int j = 0; j < n_s; ++j) rk += surv[j] > ki;
    if (rk < a.K) out_keys[rk] = ki;
  }
  if (tid == 0) {
    double stot = 0.0;
    for (int w = 0; w < kT / 32; ++w) stot += sc.red_d[w];
    a.part_m[part] = M;
    a.part_s[part] = have_mass ? stot : 0.0;
    a.part_n[part] = min(n_s, a.K);
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) sc.last = atomicAdd(&a.row_cnt[row], 1u) == (uint32_t)(a.C - 1);
  __syncthreads();
  if (!sc.last) return;
  __threadfence();

  // ---- merge of the row's chunk partials (last arriving CTA)
  const size_t part0 = (size_t)row * a.C;
  // fp64 log-sum-exp over chunks
  float Mrow = -INFINITY;
  for (int q = 0; q < a.C; ++q) Mrow = fmaxf(Mrow, __ldcg(&a.part_m[part0 + q]));
  double acc = 0.0;
  if (warp == 0) {
    for (int q = lane; q < a.C; q += 32) {
      float mq = __ldcg(&a.part_m[part0 + q]);
      double sq = __ldcg(&a.part_s[part0 + q]);
      if (mq != -INFINITY) acc += sq * exp((double)mq - (double)Mrow);
    }
    acc = warp_sum_d(acc);
  }
  // stage the sorted chunk lists in shared memory (reusing the chunk buffer)
  uint64_t *lists = reinterpret_cast<uint64_t *>(buf);
  int *offs = sc.scan;  // offs[q] = start of list q, offs[C] = total
  if (tid == 0) {
    int run = 0;
    for (int q = 0; q < a.C; ++q) { offs[q] = run; run += __ldcg(&a.part_n[part0 + q]); }
    offs[a.C] = run;
  }
  __syncthreads();
  const int total = offs[a.C];
  for (int i = tid; i < total; i += kT) {
    int q = 0;
    while (offs[q + 1] <= i) ++q;
    lists[i] = __ldcg(&a.part_keys[(part0 + q) * a.K + (i - offs[q])]);
  }
  __syncthreads();
  uint64_t *final_keys = surv;
  for (int i = tid; i < total; i += kT) {
    int q = 0;
    while (offs[q + 1] <= i) ++q;
    const uint64_t key = lists[i];
    int rk = i - offs[q];
    for (int o = 0; o < a.C && rk < a.K; ++o) {
      if (o == q) continue;
      int lo = offs[o], hi = offs[o + 1];
      while (lo < hi) {
        int mid = (lo + hi) >> 1;
        if (lists[mid] > key) lo = mid + 1; else hi = mid;
      }
      rk += lo - offs[o];
    }
    if (rk < a.K) final_keys[rk] = key;
  }
  if (tid == 0) {
    double lse = (double)Mrow + log(acc);
    sc.red_d[0] = lse;
    int st = 0;
    if (Mrow == INFINITY || !(acc == acc) || acc == INFINITY) st |= BASTION_STATUS_NONFINITE;
    if (Mrow == -INFINITY) st |= BASTION_STATUS_EMPTY_ROW;
    if (st) atomicOr(&a.status[req], st);
    a.lse[row] = lse;
    a.row_cnt[row] = 0u;
  }
  __syncthreads();
  const double lse = sc.red_d[0];
  for (int j = tid; j < a.K; j += kT) {
    const uint64_t key = final_keys[j];
    const float v = key_value(key);
    const size_t o = (size_t)row * a.K + j;
    a.topk_logit[o] = v;
    a.topk_tok[o] = (int32_t)key_token(key);
    if (a.topk_logq) a.topk_logq[o] = (float)((double)v - lse);
  }
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

struct TopkPlan {
  int CL, C;
  size_t smem;
};

TopkPlan plan_topk(int V, int K, int es) {
  TopkPlan p;
  p.CL = es == 2 ? 16384 : 8192;
  p.C = (V + p.CL - 1) / p.CL;
  while (p.C > 256 || (size_t)p.C * K * 8 > (size_t)p.CL * es) {
    p.CL *= 2;
    p.C = (V + p.CL - 1) / p.CL;
  }
  p.smem = 16 + kCap * 8 + ((sizeof(Scratch) + 127) / 128) * 128 + kPad + (size_t)p.CL * es + 32;
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
  return p.smem <= 200 * 1024;
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
  a.part_s = reinterpret_cast<double *>(w);
  w += align256(P * 8);
  a.part_n = reinterpret_cast<int32_t *>(w);
  w += align256(P * 4);
  a.part_keys = reinterpret_cast<uint64_t *>(w);
  w += align256(P * K * 8);
  a.row_cnt = reinterpret_cast<uint32_t *>(w);
  const unsigned grid = (unsigned)P;
  if (es == 4) {
    if (p.smem > 48 * 1024)
      cudaFuncSetAttribute(topk_chunk_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
    topk_chunk_kernel<4><<<grid, kT, p.smem, stream>>>(a);
  } else {
    if (p.smem > 48 * 1024)
      cudaFuncSetAttribute(topk_chunk_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
    topk_chunk_kernel<2><<<grid, kT, p.smem, stream>>>(a);
  }
  return cudaGetLastError() == cudaSuccess ? BASTION_OK : BASTION_ERR_LAUNCH;
}

}  // namespace bastion
