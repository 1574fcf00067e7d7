// Calibration of the verification cost model, on the device.
//
// Bastion (gist.science/nl/paper/2605.29727), "Methodologie" §3,
// "Latentiemodellering": T_verify(N) comes from a hardware-aware roofline model
// of memory bandwidth and compute limits, calibrated with observed runtimes to
// correct for kernel fusion and scheduling overhead.  Here the roofline of a
// target forward over N tree tokens is
//   roof(N) = max((bytes0 + bytes1 N) / bw, (flops0 + flops1 N) / peak)
// and the calibration is the least-squares line T_verify = alpha roof + beta
// through observed (N, ms) samples (alpha = 1, beta = mean(t - roof) when the
// samples' roofline values have no spread).  One CTA forms the sums in fp64
// (one pass of raw moments, no division per sample), then writes the
// controller's table C(N) = t_draft + alpha
// roof(N) + beta for N = 0 .. n_max where the tree build reads it, so a serving
// loop can refresh its cost model between steps without a host round trip.
#include "common.cuh"

namespace bastion {

namespace {

constexpr int kCT = 256;

struct CalArgs {
  const float *n, *ms;
  int count, n_max;
  double bytes0, bytes1, flops0, flops1, t_draft;  // divided by bw and peak
  float *cost, *params;
  int32_t *status;
};

// The divisions by bw and peak are folded into the constants once (the fp64
// pipe of GB300 is narrow: a division is a long instruction sequence).
__device__ __forceinline__ double roof_of(const CalArgs &a, double N) {
  return fmax(fma(a.bytes1, N, a.bytes0), fma(a.flops1, N, a.flops0));
}

// Sum of x over the CTA (every thread gets it); sh holds kCT / 32 doubles.
__device__ __forceinline__ double cta_sum(double x, double *sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(kFull, x, o);
  __syncthreads();
  if (lane == 0) sh[warp] = x;
  __syncthreads();
  double t = 0.0;
#pragma unroll
  for (int w = 0; w < kCT / 32; ++w) t += sh[w];
  return t;
}

__global__ void __launch_bounds__(kCT) calibrate_kernel(CalArgs a) {
  __shared__ double sh[kCT / 32];
  griddep_wait();
  griddep_launch_dependents();
  const int tid = threadIdx.x;
  // one pass of raw moments (in fp64 the cancellation in the centred forms
  // below costs ~1e-16 (mean / spread)^2, far below what the table needs)
  double sr = 0.0, st = 0.0, s2 = 0.0, sx = 0.0;
  int bad = 0;
  for (int k = tid; k < a.count; k += kCT) {
    const double t = a.ms[k], N = a.n[k];
    bad |= !(t == t) || !(N == N) || t == (double)INFINITY || N == (double)INFINITY;
    const double r = roof_of(a, N);
    sr += r;
    st += t;
    s2 = fma(r, r, s2);
    sx = fma(r, t, sx);
  }
  sr = cta_sum(sr, sh);
  st = cta_sum(st, sh);
  s2 = cta_sum(s2, sh);
  sx = cta_sum(sx, sh);
  bad = __syncthreads_or(bad);
  const double inv = 1.0 / a.count, mr = sr * inv, mt = st * inv;
  const double srr = s2 - sr * mr, srt = sx - sr * mt;
  double alpha = 1.0, beta = mt - mr;
  if (srr > 1e-12 * fmax(1.0, mr * mr) * a.count) {
    alpha = srt / srr;
    beta = mt - alpha * mr;
  }
  for (int N = tid; N <= a.n_max; N += kCT) {
    const double c = a.t_draft + alpha * roof_of(a, (double)N) + beta;
    a.cost[N] = (float)c;
    bad |= N >= 1 && !(c > 0.0 && c < (double)INFINITY);
  }
  bad = __syncthreads_or(bad);
  if (tid == 0) {
    a.params[0] = (float)alpha;
    a.params[1] = (float)beta;
    if (bad) atomicOr(a.status, BASTION_STATUS_BAD_COST);
  }
}

}  // namespace

int launch_calibrate(const float *sample_n, const float *sample_ms, int n_samples, double bytes0,
                     double bytes1, double flops0, double flops1, double bw, double peak,
                     double t_draft, int n_max, float *cost_ms, float *params, int32_t *status,
                     cudaStream_t stream) {
  CalArgs a;
  a.n = sample_n;
  a.ms = sample_ms;
  a.count = n_samples;
  a.n_max = n_max;
  a.bytes0 = bytes0 / bw;  // roof(N) = max(bytes0 + bytes1 N, flops0 + flops1 N) in these units
  a.bytes1 = bytes1 / bw;
  a.flops0 = flops0 / peak;
  a.flops1 = flops1 / peak;
  a.t_draft = t_draft;
  a.cost = cost_ms;
  a.params = params;
  a.status = status;
  const cudaError_t e = launch_pdl(calibrate_kernel, dim3(1), dim3(kCT), 0, stream, a);
  return (e == cudaSuccess && cudaGetLastError() == cudaSuccess) ? BASTION_OK : BASTION_ERR_LAUNCH;
}

}  // namespace bastion
