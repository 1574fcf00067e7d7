// Stochastic verification at temperature T > 0 (the next step after greedy
// verification in the draft-tree path).
//
// Bastion (gist.science/nl/paper/2605.29727) evaluates greedy decoding only
// ("Experimentele Resultaten"); DBlast (gist.science/nl/paper/2608.05448,
// introduction) argues that sampled decoding is the regime that matters.  For a
// tree of deterministic candidates the lossless reading is: every node's token
// is a draw from softmax(l / T), by inverse transform with the caller's uniform
// u in [0, 1): the smallest v whose cumulative weight sum_{w <= v} exp(l_w / T)
// exceeds u times the row's total; the greedy walk then runs over the draws.
//
// Design (HBM-bound: one read of every live row, then one 4 KB item per row):
//  * sweep: persistent warps take the 4 KB items of the live rows round robin
//    (as the greedy sweep).  Per item a lane sums 2^(l log2(e)/T - c) over
//    its elements with c = floor(m log2(e)/T) of its max m, so every exponent
//    is below ~1; the warp scales the lanes' sums to the item's largest c by
//    exact powers of two and adds them in two-float arithmetic.  The item's
//    (max, c, sum) goes to the workspace;
//  * draw: persistent warps take the live rows in turn.  A warp scales the
//    row's item sums to its largest c (exact), scans them in item order in
//    two-float arithmetic (no fp64: GB300's fp64 rate is a small fraction of
//    its fp32 rate), takes the item holding u times the total, and reads that
//    item again with all of its loads in flight at once.  In token order (head
//    elements, 8 blocks of 32 lanes x 8 elements, tail elements) it forms every
//    vector's weight first, the 8 block totals by independent reductions,
//    then scans only the block that holds the draw.  The drawn token goes to
//    the row's key in the workspace;
//  * the greedy finish kernel decodes the keys, walks the tree and resets them.
#include <cuda_bf16.h>

#include "common.cuh"

namespace bastion {

int launch_verify_finish(const int32_t *n_nodes, const int32_t *parent, const int32_t *token, int B,
                         int n_max, int b, int32_t *argmax, int32_t *accept_len, int32_t *accept_nodes,
                         int32_t *out_tokens, uint64_t *row_key, int32_t *status, cudaStream_t stream);

namespace {

constexpr int kST = 256;  // threads per CTA
constexpr int kSW = kST / 32;
constexpr int kSV = 8;    // 16-byte vectors per lane per item
constexpr float kL2e = 1.4426950216293335f;
constexpr float kCNone = -1.0e30f;

struct SampleArgs {
  const unsigned char *logits;
  int B, n_max, V, SEG, nseg;
  int64_t ld;
  float l2et;  // log2(e) / T
  const double *u;
  const int32_t *n_nodes;
  float4 *part;       // [B * n_max * nseg] an item's (max, c, sum hi, sum lo)
  uint64_t *row_key;  // [B * n_max] the drawn token, as a greedy row key
  int32_t *status;
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float pow2_int(float d) {
  return d < -126.f ? 0.f : __int_as_float(((int)d + 127) << 23);
}
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

template <int ES>
__device__ __forceinline__ float elem_at(const unsigned char *p) {
  if constexpr (ES == 4) return *reinterpret_cast<const float *>(p);
  else return __uint_as_float((uint32_t)(*reinterpret_cast<const uint16_t *>(p)) << 16);
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

// Where item sg of row (r, i) lies: first element g0, 16-byte aligned middle
// (vp, nvec vectors) between nh head and n - t0 tail elements.
struct Item {
  int e0, n, nh, t0, nvec;
  const unsigned char *g0;
  const uint4 *vp;
};
template <int ES>
__device__ __forceinline__ Item item_of(const SampleArgs &a, int r, int i, int sg) {
  Item t;
  t.e0 = sg * a.SEG;
  t.n = min(a.V - t.e0, a.SEG);
  t.g0 = a.logits + (((size_t)r * a.n_max + i) * (size_t)a.ld + t.e0) * ES;
  const uintptr_t ga0 = ((uintptr_t)t.g0 + 15) & ~(uintptr_t)15;
  const uintptr_t ga1 = ((uintptr_t)t.g0 + (uintptr_t)t.n * ES) & ~(uintptr_t)15;
  const int body = ga1 > ga0 ? (int)(ga1 - ga0) : 0;
  t.nh = body ? (int)(ga0 - (uintptr_t)t.g0) / ES : t.n;
  t.t0 = t.nh + body / ES;
  t.nvec = body / 16;
  t.vp = reinterpret_cast<const uint4 *>(ga0);
  return t;
}

// The scalar element lane j of an item holds, or -1: head j < nh first, then
// the tail.
__device__ __forceinline__ int scalar_of(const Item &t, int j) {
  return j < t.nh ? j : (j - t.nh < t.n - t.t0 ? t.t0 + (j - t.nh) : -1);
}

// Weight 2^(x l2et - c) of a logit; -inf gives 0.
__device__ __forceinline__ float weight(float x, float l2et, float c) { return ex2(fmaf(x, l2et, -c)); }

template <int ES>
__device__ __forceinline__ uint4 neg_inf_vec() {
  return ES == 2 ? make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u)
                 : make_uint4(0xff800000u, 0xff800000u, 0xff800000u, 0xff800000u);
}

// Max over a lane's kSV vectors (NaN ignored): one chain of packed maxima.
template <int ES>
__device__ __forceinline__ float lane_max(const uint4 (&x)[kSV]) {
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
    float m = -INFINITY;
#pragma unroll
    for (int u = 0; u < kSV; ++u)
      m = fmaxf(fmaxf(m, fmaxf(__uint_as_float(x[u].x), __uint_as_float(x[u].y))),
                fmaxf(__uint_as_float(x[u].z), __uint_as_float(x[u].w)));
    return m;
  }
}

// Sum of 2^(x l2et + nc) over a lane's kSV vectors: packed FMAs and adds.
template <int ES>
__device__ __forceinline__ float lane_weight_sum(const uint4 (&x)[kSV], float l2et, float nc) {
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
          : "f"(f[i]), "f"(f[i + 1]), "f"(f[i + 2]), "f"(f[i + 3]), "f"(nc), "f"(l2et));
      const float e0 = ex2(t0), e1 = ex2(t1), e2 = ex2(t2), e3 = ex2(t3);
      asm("{\n .reg .b64 a, b, p, q;\n mov.b64 a, {%0, %1};\n mov.b64 b, {%2, %3};\n"
          " mov.b64 p, {%4, %5};\n mov.b64 q, {%6, %7};\n"
          " add.rn.f32x2 a, a, p;\n add.rn.f32x2 b, b, q;\n"
          " mov.b64 {%0, %1}, a;\n mov.b64 {%2, %3}, b;\n}\n"
          : "+f"(s0), "+f"(s1), "+f"(s2), "+f"(s3)
          : "f"(e0), "f"(e1), "f"(e2), "f"(e3));
    }
  }
  const float2 p = two_sum(s0 + s1, s2 + s3);
  return p.x + p.y;
}

// Exclusive prefix over requests of per-request counts (valid n_nodes times
// per_row) into prefix[0..B]; every CTA computes the same.
__device__ __forceinline__ void request_prefix(const int32_t *n_nodes, int B, int n_max, int per_row,
                                               int *prefix, int *s_tot) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (B + kST - 1) / kST;
  const int r0 = min(B, tid * per), r1 = min(B, r0 + per);
  int sum = 0;
  for (int r = r0; r < r1; ++r) {
    const int nn = n_nodes[r];
    sum += (nn >= 1 && nn <= n_max) ? nn * per_row : 0;
  }
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s_tot[warp] = incl;
  __syncthreads();
  int run = incl - sum;
  for (int w = 0; w < warp; ++w) run += s_tot[w];
  for (int r = r0; r < r1; ++r) {
    prefix[r] = run;
    const int nn = n_nodes[r];
    run += (nn >= 1 && nn <= n_max) ? nn * per_row : 0;
  }
  if (r1 == B && r0 < r1) prefix[B] = run;
  __syncthreads();
}

template <int ES>
__global__ void __launch_bounds__(kST, 4) sample_sweep_kernel(SampleArgs a) {
  extern __shared__ int prefix[];  // [B + 1]
  __shared__ int s_tot[kSW];
  const int lane = threadIdx.x & 31;
  griddep_wait();
  griddep_launch_dependents();
  request_prefix(a.n_nodes, a.B, a.n_max, a.nseg, prefix, s_tot);
  const int total = prefix[a.B];
  const int gw = blockIdx.x * kSW + (threadIdx.x >> 5), nw = gridDim.x * kSW;
  // items dealt to the warps round robin: the grid reads one contiguous window
  for (int item = gw; item < total; item += nw) {
    // the item's request (binary search of the prefix), row and segment
    int lo = 0, hi = a.B;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (prefix[mid] <= item) lo = mid; else hi = mid;
    }
    const int r = lo;
    const int off = item - prefix[r];
    const int i = off / a.nseg;
    const int sg = off - i * a.nseg;
    const Item t = item_of<ES>(a, r, i, sg);
    uint4 x[kSV];
#pragma unroll
    for (int u = 0; u < kSV; ++u) {
      const int v = lane + 32 * u;
      x[u] = v < t.nvec ? ld_stream_v4(t.vp + v) : neg_inf_vec<ES>();
    }
    const int e = scalar_of(t, lane);
    const float xs = e >= 0 ? elem_at<ES>(t.g0 + (size_t)e * ES) : -INFINITY;
    const float m = fmaxf(lane_max<ES>(x), xs);
    const float c = m > -INFINITY ? (m < INFINITY ? floorf(m * a.l2et) : INFINITY) : kCNone;
    float s = lane_weight_sum<ES>(x, a.l2et, -c);
    if (e >= 0) s += weight(xs, a.l2et, c);
    // the item: max, its largest c, and the lanes' sums scaled to it
    const float M = warp_max_f(m), cI = warp_max_f(c);
    const float f = c > kCNone ? pow2_int(c - cI) : 0.f;
    float2 S = make_float2(s * f, 0.f);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
      S = ff_add(S, make_float2(__shfl_xor_sync(kFull, S.x, o), __shfl_xor_sync(kFull, S.y, o)));
    if (lane == 0) a.part[((size_t)r * a.n_max + i) * a.nseg + sg] = make_float4(M, cI, S.x, S.y);
  }
}

constexpr int kCacheP = 4;  // item results a lane of the draw kernel keeps in registers

// Item q (the lane's k-th): from the registers when cached, else from L2.
__device__ __forceinline__ float4 part_at(const float4 (&pc)[kCacheP], const float4 *pp, int q, int k) {
  float4 p = pc[0];
#pragma unroll
  for (int j = 1; j < kCacheP; ++j)
    if (k == j) p = pc[j];
  return k < kCacheP ? p : __ldcg(pp + q);
}

// a > b for normalised two-float values.
__device__ __forceinline__ bool ff_gt(float2 a, float2 b) { return a.x > b.x || (a.x == b.x && a.y > b.y); }

// Inclusive scan of a float over the warp's lanes.
__device__ __forceinline__ float warp_incl_scan(float v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(kFull, v, o);
    if (lane >= o) v += y;
  }
  return v;
}

// One warp per live row: the draw by inverse transform.
template <int ES>
__device__ __forceinline__ void draw_row(const SampleArgs &a, int r, int i, int lane) {
  constexpr int NE = 16 / ES;
  const int w = r * a.n_max + i;
  const double ud = a.u[w];  // loaded with the items' results
  const float4 *pp = a.part + (size_t)w * a.nseg;
  const int P = (a.nseg + 31) / 32;  // items per lane, contiguous
  float4 pc[kCacheP];                // the first kCacheP of them, loaded once
#pragma unroll
  for (int k = 0; k < kCacheP; ++k) {
    const int q = lane * P + k;
    pc[k] = k < P && q < a.nseg ? __ldcg(pp + q) : make_float4(-INFINITY, kCNone, 0.f, 0.f);
  }
  float M = -INFINITY, cR = kCNone;
  for (int k = 0; k < P; ++k) {
    const int q = lane * P + k;
    if (q < a.nseg) {
      const float4 p = part_at(pc, pp, q, k);
      M = fmaxf(M, p.x);
      cR = fmaxf(cR, p.y);
    }
  }
  M = warp_max_f(M);
  cR = warp_max_f(cR);
  // the lane's items in order, scaled to cR (exact powers of two)
  float2 ls = make_float2(0.f, 0.f);
  for (int k = 0; k < P; ++k) {
    const int q = lane * P + k;
    if (q < a.nseg) {
      const float4 p = part_at(pc, pp, q, k);
      const float f = p.y > kCNone ? pow2_int(p.y - cR) : 0.f;
      ls = ff_add(ls, make_float2(p.z * f, p.w * f));
    }
  }
  float2 inc = ls;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float2 y = make_float2(__shfl_up_sync(kFull, inc.x, o), __shfl_up_sync(kFull, inc.y, o));
    if (lane >= o) inc = ff_add(y, inc);
  }
  const float2 total = make_float2(__shfl_sync(kFull, inc.x, 31), __shfl_sync(kFull, inc.y, 31));
  int st = 0;
  if (M == INFINITY || !(total.x == total.x) || total.x == INFINITY || !(cR < INFINITY))
    st |= BASTION_STATUS_NONFINITE;
  if (!(total.x > 0.f)) st |= BASTION_STATUS_EMPTY_ROW;
  if (st) {
    if (lane == 0) {
      atomicOr(&a.status[r], st);
      a.row_key[w] = make_key(0.f, 0u);
    }
    return;
  }
  // t = u * total in two-float arithmetic (the only double is the uniform)
  float2 t;
  {
    const float uh = (float)ud, ul = (float)(ud - (double)uh);
    const float th = uh * total.x;
    t = two_sum(th, fmaf(uh, total.x, -th) + (uh * total.y + ul * total.x));
  }
  // the lane, then the item, holding t
  float2 ex = make_float2(__shfl_up_sync(kFull, inc.x, 1), __shfl_up_sync(kFull, inc.y, 1));
  if (lane == 0) ex = make_float2(0.f, 0.f);
  const unsigned over = __ballot_sync(kFull, ff_gt(inc, t));
  // rounding may leave t at the total: then the last lane with weight
  const int L = over ? __ffs(over) - 1 : 31 - __clz(__ballot_sync(kFull, ls.x > 0.f) | 1u);
  int q = -1;
  float cq = kCNone;
  float2 res = make_float2(0.f, 0.f);
  if (lane == L) {
    float2 cum = ex;
    for (int k = 0; k < P; ++k) {
      const int qq = lane * P + k;
      if (qq >= a.nseg) break;
      const float4 p = part_at(pc, pp, qq, k);
      const float f = p.y > kCNone ? pow2_int(p.y - cR) : 0.f;
      const float2 wq = make_float2(p.z * f, p.w * f);
      if (wq.x > 0.f) {  // the last item with weight, should rounding pass the end
        q = qq;
        cq = p.y;
        res = ff_add(t, make_float2(-cum.x, -cum.y));
      }
      const float2 nc = ff_add(cum, wq);
      if (ff_gt(nc, t)) break;
      cum = nc;
    }
  }
  q = __shfl_sync(kFull, q, L);
  cq = __shfl_sync(kFull, cq, L);
  const float resf = __shfl_sync(kFull, res.x + res.y, L);
  if (q < 0) q = 0;
  // the item again, in token order, in units of its own c (an exact power of
  // two away); all of its loads (head, middle, tail) are issued before any is
  // used
  const float dq = cR - cq;  // >= 0, <= 126 for an item with weight
  float rem = dq <= 126.f ? resf * __int_as_float(((int)dq + 127) << 23) : 0.f;
  const Item it = item_of<ES>(a, r, i, q);
  const int eh = lane < it.nh ? lane : -1;
  const int et = lane < it.n - it.t0 ? it.t0 + lane : -1;
  uint4 xv[kSV];
#pragma unroll
  for (int u = 0; u < kSV; ++u) {
    const int v = lane + 32 * u;
    xv[u] = v < it.nvec ? ld_stream_v4(it.vp + v) : neg_inf_vec<ES>();
  }
  const float xh = eh >= 0 ? elem_at<ES>(it.g0 + (size_t)eh * ES) : -INFINITY;
  const float xt = et >= 0 ? elem_at<ES>(it.g0 + (size_t)et * ES) : -INFINITY;
  int y = -1, last = -1;
  {  // head elements
    const float wv = eh >= 0 ? weight(xh, a.l2et, cq) : 0.f;
    const float incl = warp_incl_scan(wv, lane);
    if (wv > 0.f) last = max(last, eh);
    const unsigned hit = __ballot_sync(kFull, incl > rem && wv > 0.f);
    if (hit) y = __ffs(hit) - 1;
    rem -= __shfl_sync(kFull, incl, 31);
  }
  if (y < 0) {
    // the middle: every vector's weight first (independent), then the block
    // of 32 vectors holding rem, then the lane, then the element
    float vsu[kSV], bt[kSV];
#pragma unroll
    for (int u = 0; u < kSV; ++u) {
      float f[NE];
      unpack<ES>(xv[u], f);
      float vs = 0.f;
#pragma unroll
      for (int k = 0; k < NE; ++k) {
        const float wk = weight(f[k], a.l2et, cq);
        vs += wk;
        if (wk > 0.f) last = max(last, it.nh + (lane + 32 * u) * NE + k);
      }
      vsu[u] = vs;
    }
#pragma unroll
    for (int u = 0; u < kSV; ++u) {
      float t2 = vsu[u];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) t2 += __shfl_xor_sync(kFull, t2, o);
      bt[u] = t2;
    }
    int ub = -1;
    float before = 0.f;
#pragma unroll
    for (int u = 0; u < kSV; ++u) {
      if (ub < 0) {
        if (bt[u] > 0.f && before + bt[u] > rem) ub = u;
        else before += bt[u];
      }
    }
    if (ub >= 0) {
      float vs = vsu[0];
      uint4 xb = xv[0];
#pragma unroll
      for (int u = 1; u < kSV; ++u)
        if (u == ub) {
          vs = vsu[u];
          xb = xv[u];
        }
      const float r2 = rem - before;
      const float incl = warp_incl_scan(vs, lane);
      unsigned hit = __ballot_sync(kFull, incl > r2 && vs > 0.f);
      if (!hit) hit = 1u << (31 - __clz(__ballot_sync(kFull, vs > 0.f)));  // rounding: the last lane with weight
      const int hl = __ffs(hit) - 1;
      if (lane == hl) {
        // the first element whose cumulative weight passes r2, else (rounding)
        // the last element with weight; static indices only
        float f[NE];
        unpack<ES>(xb, f);
        float cum = incl - vs;
        int kf = -1, kl = 0;
#pragma unroll
        for (int k = 0; k < NE; ++k) {
          const float wk = weight(f[k], a.l2et, cq);
          if (kf < 0 && wk > 0.f && cum + wk > r2) kf = k;
          if (wk > 0.f) kl = k;
          cum += wk;
        }
        y = it.nh + (lane + 32 * ub) * NE + (kf >= 0 ? kf : kl);
      }
      y = __shfl_sync(kFull, y, hl);
    } else {
      rem -= before;
    }
  }
  if (y < 0) {  // tail elements
    const float wv = et >= 0 ? weight(xt, a.l2et, cq) : 0.f;
    const float incl = warp_incl_scan(wv, lane);
    if (wv > 0.f) last = max(last, et);
    const unsigned hit = __ballot_sync(kFull, incl > rem && wv > 0.f);
    if (hit) y = __shfl_sync(kFull, et, __ffs(hit) - 1);
  }
  last = __reduce_max_sync(kFull, (unsigned)(last + 1)) - 1;
  if (y < 0) y = last >= 0 ? last : 0;
  if (lane == 0) a.row_key[w] = make_key(0.f, (uint32_t)(it.e0 + y));
}

// A persistent grid whose warps take the live rows in turn.
template <int ES>
__global__ void __launch_bounds__(kST, 2) sample_find_kernel(SampleArgs a) {
  extern __shared__ int prefix[];  // [B + 1] live rows before each request
  __shared__ int s_tot[kSW];
  const int lane = threadIdx.x & 31;
  griddep_wait();
  griddep_launch_dependents();
  request_prefix(a.n_nodes, a.B, a.n_max, 1, prefix, s_tot);
  const int total = prefix[a.B];
  const int nw = gridDim.x * kSW;
  for (int g = blockIdx.x * kSW + (threadIdx.x >> 5); g < total; g += nw) {
    int lo = 0, hi = a.B;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (prefix[mid] <= g) lo = mid; else hi = mid;
    }
    draw_row<ES>(a, lo, g - prefix[lo], lane);
  }
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }
int sample_items(int V, int es) { return (V + 32 * kSV * (16 / es) - 1) / (32 * kSV * (16 / es)); }

}  // namespace

size_t verify_sample_workspace_bytes(int B, int n_max, int V) {
  return align256((size_t)B * n_max * 8) + align256((size_t)B * n_max * sample_items(V, 4) * 16);
}

int launch_verify_sample(const void *target, int dtype, int B, int n_max, int V, int64_t ld, int b,
                         float temperature, const double *uniforms, const int32_t *n_nodes,
                         const int32_t *parent, const int32_t *token, int32_t *sampled,
                         int32_t *accept_len, int32_t *accept_nodes, int32_t *out_tokens, void *ws,
                         int32_t *status, cudaStream_t stream) {
  const int es = dtype == BASTION_F32 ? 4 : 2;
  SampleArgs a;
  a.logits = static_cast<const unsigned char *>(target);
  a.B = B;
  a.n_max = n_max;
  a.V = V;
  a.SEG = 32 * kSV * (16 / es);
  a.nseg = sample_items(V, es);
  a.ld = ld;
  a.l2et = kL2e / temperature;
  a.u = uniforms;
  a.n_nodes = n_nodes;
  unsigned char *w = static_cast<unsigned char *>(ws);
  a.row_key = reinterpret_cast<uint64_t *>(w);
  a.part = reinterpret_cast<float4 *>(w + align256((size_t)B * n_max * 8));
  a.status = status;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const size_t smem = (size_t)(B + 1) * 4;
  auto sweep = es == 4 ? sample_sweep_kernel<4> : sample_sweep_kernel<2>;
  auto find = es == 4 ? sample_find_kernel<4> : sample_find_kernel<2>;
  int per_sm = 1;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, sweep, kST, smem);
  if (per_sm < 1) per_sm = 1;
  long long grid = (long long)sms * per_sm;
  const long long max_ctas = ((long long)B * n_max * a.nseg + kSW - 1) / kSW;
  if (grid > max_ctas) grid = max_ctas;
  if (grid < 1) grid = 1;
  cudaError_t e = launch_pdl(sweep, dim3((unsigned)grid), dim3(kST), smem, stream, a);
  if (e == cudaSuccess) {
    int fsm = 1;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&fsm, find, kST, smem);
    long long fgrid = (long long)sms * (fsm < 1 ? 1 : fsm);
    const long long fmax = ((long long)B * n_max + kSW - 1) / kSW;
    if (fgrid > fmax) fgrid = fmax;
    e = launch_pdl(find, dim3((unsigned)fgrid), dim3(kST), smem, stream, a);
  }
  if (e != cudaSuccess || cudaGetLastError() != cudaSuccess) return BASTION_ERR_LAUNCH;
  return launch_verify_finish(n_nodes, parent, token, B, n_max, b, sampled, accept_len, accept_nodes,
                              out_tokens, a.row_key, status, stream);
}

}  // namespace bastion
