// Step 4 of the draft-tree path: greedy (temperature 0) verification.
//
// Bastion (gist.science/nl/paper/2605.29727), "Experimentele Resultaten": the
// evaluation decodes greedily.  The target's greedy token at every tree node is
// the argmax of that node's target logits (ties: lowest token); the longest root
// path whose tokens match the greedy tokens of their parents is accepted, and
// the greedy token at its end is the bonus token.
//
// Design (HBM-bound sweep over sum_r n_nodes[r] rows of V logits):
//  * persistent grid (as many CTAs per SM as fit); the work items are (request, node row,
//    vocab chunk) with the row count per request read on the device, so only
//    rows < n_nodes[r] are ever read;
//  * a chunk is streamed with 16-byte non-allocating loads, 4 in flight per
//    thread; each thread keeps the max value and the index of the vector that
//    first reached it (packed bf16x2 max, NaN-propagating), then re-reads that
//    one vector to find the lowest token holding the max;
//  * the chunk winner (value desc, token asc as one 64-bit key) is merged with
//    atomicMax into the row's key in the workspace;
//  * the last CTA to finish a request's items (arrival counter, no waiting)
//    decodes the argmaxes, runs the accept walk from the root and resets the
//    request's workspace entries to zero.
#include "common.cuh"

namespace bastion {

namespace {

constexpr int kVT = 256;
constexpr int kUnroll = 4;

struct VerifyArgs {
  const unsigned char *logits;
  int B, n_max, V, b, CL, Cv;
  int64_t ld;
  const int32_t *n_nodes, *parent, *token;
  int32_t *argmax, *accept_len, *accept_nodes, *out_tokens;
  uint64_t *row_key;
  uint32_t *req_cnt;
  int32_t *status;
};

template <int ES>
__device__ __forceinline__ float vmax_nan(const uint4 &x) {
  if constexpr (ES == 4) {
    float a, c, m;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(a) : "f"(__uint_as_float(x.x)), "f"(__uint_as_float(x.y)));
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(c) : "f"(__uint_as_float(x.z)), "f"(__uint_as_float(x.w)));
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(m) : "f"(a), "f"(c));
    return m;
  } else {
    uint32_t a, c, m;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(a) : "r"(x.x), "r"(x.y));
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(c) : "r"(x.z), "r"(x.w));
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(m) : "r"(a), "r"(c));
    float lo = bf16lo(m), hi = bf16hi(m), r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(lo), "f"(hi));
    return r;
  }
}

template <int ES>
__device__ __forceinline__ float elem_of(const uint4 &x, int i) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
  if constexpr (ES == 4) return __uint_as_float(w[i]);
  else return (i & 1) ? bf16hi(w[i >> 1]) : bf16lo(w[i >> 1]);
}

template <int ES>
__device__ __forceinline__ float load_elem_g(const unsigned char *p) {
  if constexpr (ES == 4) return *reinterpret_cast<const float *>(p);
  else return __uint_as_float((uint32_t)(*reinterpret_cast<const uint16_t *>(p)) << 16);
}

// better(a, b): a has a larger value, or a is NaN and b is not.
__device__ __forceinline__ bool takes_over(float a, float b) { return a > b || (a != a && b == b); }

template <int ES>
__global__ void __launch_bounds__(kVT) verify_kernel(VerifyArgs a) {
  extern __shared__ int prefix[];  // [B + 1]
  __shared__ uint64_t red[kVT / 32];
  __shared__ int s_last;
  __shared__ int s_am[256], s_par[256], s_tok[256];
  __shared__ int s_tot[kVT / 32];

  constexpr int NE = 16 / ES;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // per-request item counts -> exclusive prefix (every CTA computes the same)
  {
    const int per = (a.B + kVT - 1) / kVT;
    const int r0 = min(a.B, tid * per), r1 = min(a.B, r0 + per);
    int sum = 0;
    for (int r = r0; r < r1; ++r) {
      const int nn = a.n_nodes[r];
      sum += (nn >= 1 && nn <= a.n_max) ? nn * a.Cv : 0;
    }
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) s_tot[warp] = incl;
    __syncthreads();
    int wbase = 0;
    for (int w = 0; w < warp; ++w) wbase += s_tot[w];
    int run = wbase + incl - sum;
    for (int r = r0; r < r1; ++r) {
      prefix[r] = run;
      const int nn = a.n_nodes[r];
      run += (nn >= 1 && nn <= a.n_max) ? nn * a.Cv : 0;
    }
    if (r1 == a.B && r0 < r1) prefix[a.B] = run;
    if (a.B == 0 && tid == 0) prefix[0] = 0;
    __syncthreads();
  }
  // requests whose n_nodes is out of range: flag and write empty results
  if (blockIdx.x == 0) {
    for (int r = tid; r < a.B; r += kVT) {
      const int nn = a.n_nodes[r];
      if (nn < 1 || nn > a.n_max) {
        atomicOr(&a.status[r], BASTION_STATUS_BAD_TREE);
        a.accept_len[r] = 0;
        for (int k = 0; k <= a.b; ++k) {
          a.accept_nodes[(size_t)r * (a.b + 1) + k] = -1;
          a.out_tokens[(size_t)r * (a.b + 1) + k] = -1;
        }
      }
    }
  }
  const int total = prefix[a.B];

  for (int item = blockIdx.x; item < total; item += gridDim.x) {
    int lo = 0, hi = a.B;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (prefix[mid] <= item) lo = mid; else hi = mid;
    }
    const int r = lo;
    const int off = item - prefix[r];
    const int i = off / a.Cv, c = off - i * a.Cv;
    const int e0 = c * a.CL;
    const int n = min(a.V - e0, a.CL);
    const unsigned char *g0 = a.logits + (((size_t)r * a.n_max + i) * (size_t)a.ld + e0) * ES;
    const uintptr_t ga0 = ((uintptr_t)g0 + 15) & ~(uintptr_t)15;
    const uintptr_t ga1 = ((uintptr_t)g0 + (uintptr_t)n * ES) & ~(uintptr_t)15;
    const int body = ga1 > ga0 ? (int)(ga1 - ga0) : 0;
    const int nh = body ? (int)(ga0 - (uintptr_t)g0) / ES : n;
    const int t0 = nh + body / ES;
    const int nvec = body / 16;
    const uint4 *vp = reinterpret_cast<const uint4 *>(ga0);

    float bv = -INFINITY;
    int bvec = -1;
    for (int v0 = tid; v0 < nvec; v0 += kVT * kUnroll) {
      uint4 x[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int v = v0 + u * kVT;
        if (v < nvec) x[u] = ld_stream_v4(vp + v);
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int v = v0 + u * kVT;
        if (v < nvec) {
          const float m = vmax_nan<ES>(x[u]);
          if (takes_over(m, bv)) { bv = m; bvec = v; }
        }
      }
    }
    uint64_t key = 0ull;
    if (bvec >= 0) {
      const uint4 x = ld_stream_v4(vp + bvec);
#pragma unroll
      for (int q = NE - 1; q >= 0; --q) {
        const float f = elem_of<ES>(x, q);
        if (f == bv || (f != f && bv != bv)) key = make_key(f, (uint32_t)(e0 + nh + bvec * NE + q));
      }
    }
    // unaligned head / tail elements
    const int nscal = nh + (n - t0);
    for (int j = tid; j < nscal; j += kVT) {
      const int e = j < nh ? j : t0 + (j - nh);
      const float f = load_elem_g<ES>(g0 + (size_t)e * ES);
      const uint64_t k2 = make_key(f, (uint32_t)(e0 + e));
      if (k2 > key) key = k2;
    }
    key = warp_max_u64(key);
    if (lane == 0) red[warp] = key;
    __syncthreads();
    if (tid == 0) {
      uint64_t m = red[0];
      for (int w = 1; w < kVT / 32; ++w) m = red[w] > m ? red[w] : m;
      atomicMax(reinterpret_cast<unsigned long long *>(&a.row_key[(size_t)r * a.n_max + i]),
                (unsigned long long)m);
      __threadfence();
      const uint32_t want = (uint32_t)(a.n_nodes[r] * a.Cv);
      s_last = atomicAdd(&a.req_cnt[r], 1u) == want - 1u;
    }
    __syncthreads();
    if (s_last) {
      __threadfence();
      const int nn = a.n_nodes[r];
      int bad = 0;
      for (int q = tid; q < nn; q += kVT) {
        const size_t o = (size_t)r * a.n_max + q;
        const uint64_t k = __ldcg(&a.row_key[o]);
        a.row_key[o] = 0ull;
        const int t = (int)key_token(k);
        const float v = key_value(k);
        bad |= (v != v) || v == INFINITY;
        s_am[q] = t;
        a.argmax[o] = t;
        s_par[q] = a.parent[o];
        s_tok[q] = a.token[o];
      }
      if (__syncthreads_or(bad) && tid == 0) atomicOr(&a.status[r], BASTION_STATUS_NONFINITE);
      if (warp == 0) {
        int32_t *an = a.accept_nodes + (size_t)r * (a.b + 1);
        int32_t *ot = a.out_tokens + (size_t)r * (a.b + 1);
        int cur = 0, len = 0;
        if (lane == 0) an[0] = 0;
        while (true) {
          const int t = s_am[cur];
          unsigned found = 0xffffffffu;
          for (int q = 1 + lane; q < nn; q += 32)
            if (s_par[q] == cur && s_tok[q] == t && (unsigned)q < found) found = (unsigned)q;
          found = __reduce_min_sync(kFull, found);
          if (found == 0xffffffffu || len >= a.b) break;
          if (lane == 0) { ot[len] = t; an[len + 1] = (int)found; }
          ++len;
          cur = (int)found;
        }
        if (lane == 0) {
          ot[len] = s_am[cur];
          for (int k = len + 1; k <= a.b; ++k) { ot[k] = -1; an[k] = -1; }
          a.accept_len[r] = len;
          a.req_cnt[r] = 0u;
        }
      }
      __syncthreads();
    }
  }
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

void plan_chunks(int V, int es, int &CL, int &Cv) {
  const int cl_max = es == 2 ? 16384 : 8192;
  Cv = (V + cl_max - 1) / cl_max;
  CL = (V + Cv - 1) / Cv;
  CL = (CL + 7) & ~7;
}

}  // namespace

size_t verify_workspace_bytes(int B, int n_max) {
  return align256((size_t)B * n_max * 8) + align256((size_t)B * 4);
}

int launch_verify(const void *target, int dtype, int B, int n_max, int V, int64_t ld, int b,
                  const int32_t *n_nodes, const int32_t *parent, const int32_t *token,
                  int32_t *argmax, int32_t *accept_len, int32_t *accept_nodes,
                  int32_t *out_tokens, void *ws, int32_t *status, cudaStream_t stream) {
  const int es = dtype == BASTION_F32 ? 4 : 2;
  VerifyArgs a;
  a.logits = static_cast<const unsigned char *>(target);
  a.B = B;
  a.n_max = n_max;
  a.V = V;
  a.b = b;
  plan_chunks(V, es, a.CL, a.Cv);
  a.ld = ld;
  a.n_nodes = n_nodes;
  a.parent = parent;
  a.token = token;
  a.argmax = argmax;
  a.accept_len = accept_len;
  a.accept_nodes = accept_nodes;
  a.out_tokens = out_tokens;
  unsigned char *w = static_cast<unsigned char *>(ws);
  a.row_key = reinterpret_cast<uint64_t *>(w);
  a.req_cnt = reinterpret_cast<uint32_t *>(w + align256((size_t)B * n_max * 8));
  a.status = status;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const size_t smem = (size_t)(B + 1) * 4;
  int per_sm = 1;
  if (es == 4)
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, verify_kernel<4>, kVT, smem);
  else
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, verify_kernel<2>, kVT, smem);
  if (per_sm < 1) per_sm = 1;
  const long long max_items = (long long)B * n_max * a.Cv;
  long long grid = (long long)sms * per_sm;
  if (grid > max_items) grid = max_items;
  if (grid < 1) grid = 1;
  if (es == 4)
    verify_kernel<4><<<(unsigned)grid, kVT, smem, stream>>>(a);
  else
    verify_kernel<2><<<(unsigned)grid, kVT, smem, stream>>>(a);
  return cudaGetLastError() == cudaSuccess ? BASTION_OK : BASTION_ERR_LAUNCH;
}

}  // namespace bastion
