// Step 4 of the draft-tree path: greedy (temperature 0) verification.
//
// Bastion (gist.science/nl/paper/2605.29727), "Experimentele Resultaten": the
// evaluation decodes greedily.  The target's greedy token at every tree node is
// the argmax of that node's target logits (ties: lowest token); the longest root
// path whose tokens match the greedy tokens of their parents is accepted, and
// the greedy token at its end is the bonus token.
//
// Design (HBM-bound sweep over sum_r n_nodes[r] rows of V logits), two kernels
// chained with programmatic dependent launch:
//  * sweep: persistent grid sized from the occupancy; the items are dealt to
//    the warps round robin (grid-stride), with no barrier and no waiting on
//    other warps.  An item is one 4 KB segment of one tree row (row counts
//    are read on the device, so only rows < n_nodes[r] are read).  A lane
//    issues its 8 x 16-byte non-allocating loads at once, keeps the running
//    max (NaN-propagating packed bf16x2 max)
//    and the first vector that reached it, then finds the lowest token holding
//    the max in that vector from the registers it already holds.  The segment
//    winner (value desc, token asc as one 64-bit key, two redux.sync
//    reductions) is merged into the row's key by a fire-and-forget 64-bit
//    atomicMax;
//  * finish: one warp per request decodes the row keys into argmaxes, runs the
//    accept walk from the root (warp-parallel child search per step) and
//    resets the keys to zero for the next call.
#include <cuda_bf16.h>

#include "common.cuh"

namespace bastion {

namespace {

constexpr int kVT = 256;             // threads per CTA
constexpr int kWarps = kVT / 32;
constexpr int kVecPerLane = 8;       // 16-byte vectors per lane per segment

struct VerifyArgs {
  const unsigned char *logits;
  int B, n_max, V, b, SEG, nseg;
  int64_t ld;
  const int32_t *n_nodes, *parent, *token;
  int32_t *argmax, *accept_len, *accept_nodes, *out_tokens;
  uint64_t *row_key;
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
  if constexpr (ES == 4) {
    const uint32_t w = i == 0 ? x.x : i == 1 ? x.y : i == 2 ? x.z : x.w;
    return __uint_as_float(w);
  } else {
    const uint32_t w = i < 2 ? x.x : i < 4 ? x.y : i < 6 ? x.z : x.w;
    return (i & 1) ? bf16hi(w) : bf16lo(w);
  }
}

template <int ES>
__device__ __forceinline__ float load_elem_g(const unsigned char *p) {
  if constexpr (ES == 4) return *reinterpret_cast<const float *>(p);
  else return __uint_as_float((uint32_t)(*reinterpret_cast<const uint16_t *>(p)) << 16);
}

// Bit i set iff element i of the vector equals v (float equality; a NaN v
// matches NaN elements).  Element 2w is the low half of word w.
template <int ES>
__device__ __forceinline__ uint32_t eq_mask(const uint4 &x, float v) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
  uint32_t m = 0;
  if (v != v) {
#pragma unroll
    for (int i = 0; i < 16 / ES; ++i) {
      const float f = elem_of<ES>(x, i);
      m |= (f != f ? 1u : 0u) << i;
    }
    return m;
  }
  if constexpr (ES == 4) {
#pragma unroll
    for (int i = 0; i < 4; ++i) m |= (__uint_as_float(w[i]) == v ? 1u : 0u) << i;
  } else {
    const __nv_bfloat162 vv = __float2bfloat162_rn(v);  // v is a bf16 value: exact
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t e = __heq2_mask(*reinterpret_cast<const __nv_bfloat162 *>(&w[i]), vv);
      m |= ((e & 1u) << (2 * i)) | (((e >> 16) & 1u) << (2 * i + 1));
    }
  }
  return m;
}

// a takes over from b: larger, or NaN when b is not.
__device__ __forceinline__ bool takes_over(float a, float b) { return a > b || (a != a && b == b); }

template <int ES>
__global__ void __launch_bounds__(kVT) verify_kernel(VerifyArgs a) {
  extern __shared__ int prefix[];  // [B + 1]
  __shared__ int s_tot[kWarps];

  constexpr int NE = 16 / ES;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  griddep_wait();
  griddep_launch_dependents();

  // per-request item counts -> exclusive prefix (every CTA computes the same)
  {
    const int per = (a.B + kVT - 1) / kVT;
    const int r0 = min(a.B, tid * per), r1 = min(a.B, r0 + per);
    int sum = 0;
    for (int r = r0; r < r1; ++r) {
      const int nn = a.n_nodes[r];
      sum += (nn >= 1 && nn <= a.n_max) ? nn * a.nseg : 0;
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
      run += (nn >= 1 && nn <= a.n_max) ? nn * a.nseg : 0;
    }
    if (r1 == a.B && r0 < r1) prefix[a.B] = run;
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
  const int gw = blockIdx.x * kWarps + warp, nw = gridDim.x * kWarps;
  // items are dealt to the warps round robin, so that at any moment the grid
  // reads one contiguous window of the live rows (a contiguous run per warp
  // scattered the reads over the whole batch and ran ~2% slower)
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
    const int e0 = sg * a.SEG;
    const int n = min(a.V - e0, a.SEG);
    const unsigned char *g0 = a.logits + (((size_t)r * a.n_max + i) * (size_t)a.ld + e0) * ES;
    const uintptr_t ga0 = ((uintptr_t)g0 + 15) & ~(uintptr_t)15;
    const uintptr_t ga1 = ((uintptr_t)g0 + (uintptr_t)n * ES) & ~(uintptr_t)15;
    const int body = ga1 > ga0 ? (int)(ga1 - ga0) : 0;
    const int nh = body ? (int)(ga0 - (uintptr_t)g0) / ES : n;
    const int t0 = nh + body / ES;
    const int nvec = body / 16;
    const uint4 *vp = reinterpret_cast<const uint4 *>(ga0);

    uint4 x[kVecPerLane];
#pragma unroll
    for (int u = 0; u < kVecPerLane; ++u) {
      const int v = lane + 32 * u;
      x[u] = v < nvec ? ld_stream_v4(vp + v) : make_uint4(0u, 0u, 0u, 0u);
    }
    float bv = -INFINITY;
    int bu = -1;
#pragma unroll
    for (int u = 0; u < kVecPerLane; ++u) {
      if (lane + 32 * u < nvec) {
        const float m = vmax_nan<ES>(x[u]);
        if (takes_over(m, bv)) { bv = m; bu = u; }
      }
    }
    uint64_t key = 0ull;
    if (bu >= 0) {
      // the first vector that reached the max, and its first element equal to it
      uint4 xb = x[0];
#pragma unroll
      for (int u = 1; u < kVecPerLane; ++u)
        if (u == bu) xb = x[u];
      const uint32_t msk = eq_mask<ES>(xb, bv);
      const int q = __ffs(msk) - 1;
      key = make_key(elem_of<ES>(xb, q), (uint32_t)(e0 + nh + (lane + 32 * bu) * NE + q));
    }
    // unaligned head / tail elements
    const int nscal = nh + (n - t0);
    for (int j = lane; j < nscal; j += 32) {
      const int e = j < nh ? j : t0 + (j - nh);
      const uint64_t k2 = make_key(load_elem_g<ES>(g0 + (size_t)e * ES), (uint32_t)(e0 + e));
      if (k2 > key) key = k2;
    }
    key = warp_max_u64(key);
    if (lane == 0)
      atomicMax(reinterpret_cast<unsigned long long *>(&a.row_key[(size_t)r * a.n_max + i]),
                (unsigned long long)key);
  }
}

// One warp per request: argmax decode, accept walk, workspace reset.
__global__ void __launch_bounds__(256) verify_finish_kernel(VerifyArgs a) {
  __shared__ int s_am[8][256];
  __shared__ int s_par[8][256];
  __shared__ int s_tok[8][256];
  griddep_wait();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int r = blockIdx.x * 8 + warp;
  if (r >= a.B) return;
  const int nn = a.n_nodes[r];
  if (nn < 1 || nn > a.n_max) return;  // flagged by the sweep
  int bad = 0;
  for (int q = lane; q < nn; q += 32) {
    const size_t o = (size_t)r * a.n_max + q;
    const uint64_t k = a.row_key[o];
    a.row_key[o] = 0ull;
    const int t = (int)key_token(k);
    const float v = key_value(k);
    bad |= (v != v) || v == INFINITY;
    s_am[warp][q] = t;
    a.argmax[o] = t;
    s_par[warp][q] = a.parent[o];
    s_tok[warp][q] = a.token[o];
  }
  if (__any_sync(kFull, bad) && lane == 0) atomicOr(&a.status[r], BASTION_STATUS_NONFINITE);
  __syncwarp();
  int32_t *an = a.accept_nodes + (size_t)r * (a.b + 1);
  int32_t *ot = a.out_tokens + (size_t)r * (a.b + 1);
  int cur = 0, len = 0;
  if (lane == 0) an[0] = 0;
  while (true) {
    const int t = s_am[warp][cur];
    unsigned found = 0xffffffffu;
    for (int q = 1 + lane; q < nn; q += 32)
      if (s_par[warp][q] == cur && s_tok[warp][q] == t && (unsigned)q < found) found = (unsigned)q;
    found = __reduce_min_sync(kFull, found);
    if (found == 0xffffffffu || len >= a.b) break;
    if (lane == 0) { ot[len] = t; an[len + 1] = (int)found; }
    ++len;
    cur = (int)found;
  }
  if (lane == 0) {
    ot[len] = s_am[warp][cur];
    for (int k = len + 1; k <= a.b; ++k) { ot[k] = -1; an[k] = -1; }
    a.accept_len[r] = len;
  }
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

size_t verify_workspace_bytes(int B, int n_max) { return align256((size_t)B * n_max * 8); }

// The decode + walk + reset of row keys alone (the stochastic verification
// writes its drawn tokens as row keys and finishes here).
int launch_verify_finish(const int32_t *n_nodes, const int32_t *parent, const int32_t *token, int B,
                         int n_max, int b, int32_t *argmax, int32_t *accept_len, int32_t *accept_nodes,
                         int32_t *out_tokens, uint64_t *row_key, int32_t *status, cudaStream_t stream) {
  VerifyArgs a = {};
  a.B = B;
  a.n_max = n_max;
  a.b = b;
  a.n_nodes = n_nodes;
  a.parent = parent;
  a.token = token;
  a.argmax = argmax;
  a.accept_len = accept_len;
  a.accept_nodes = accept_nodes;
  a.out_tokens = out_tokens;
  a.row_key = row_key;
  a.status = status;
  const cudaError_t e = launch_pdl(verify_finish_kernel, dim3((unsigned)((B + 7) / 8)), dim3(256), 0, stream, a);
  return (e == cudaSuccess && cudaGetLastError() == cudaSuccess) ? BASTION_OK : BASTION_ERR_LAUNCH;
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
  a.SEG = 32 * kVecPerLane * (16 / es);
  a.nseg = (V + a.SEG - 1) / a.SEG;
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
  const long long max_ctas = ((long long)B * n_max * a.nseg + kWarps - 1) / kWarps;
  long long grid = (long long)sms * per_sm;
  if (grid > max_ctas) grid = max_ctas;
  if (grid < 1) grid = 1;
  cudaError_t e1 = es == 4 ? launch_pdl(verify_kernel<4>, dim3((unsigned)grid), dim3(kVT), smem, stream, a)
                           : launch_pdl(verify_kernel<2>, dim3((unsigned)grid), dim3(kVT), smem, stream, a);
  cudaError_t e2 = launch_pdl(verify_finish_kernel, dim3((unsigned)((B + 7) / 8)), dim3(256), 0, stream, a);
  return (e1 == cudaSuccess && e2 == cudaSuccess && cudaGetLastError() == cudaSuccess) ? BASTION_OK
                                                                                         : BASTION_ERR_LAUNCH;
}

}  // namespace bastion
