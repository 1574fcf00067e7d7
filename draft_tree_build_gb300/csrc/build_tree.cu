// Steps 2-3 of the draft-tree path: best-first prefix-tree expansion under the
// online budget controller, and the emitted tree arrays, as a kernel of its
// own (one CTA per request) after the top-K step.  The build itself (scores,
// frontier, stop test, outputs) is the device code of tree_build.cuh; see
// there for the design.
//
// Bastion (gist.science/nl/paper/2605.29727), Methodologie §1-§3.
#include "tree_build.cuh"

namespace bastion {

namespace {

constexpr int kTreeThreads = 128;  // staging by 4 warps; then warp 0 alone

template <int S>  // register slots per lane: S * 32 >= n_max
__global__ void __launch_bounds__(kTreeThreads) build_tree_kernel(TreeArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int r = blockIdx.x, tid = threadIdx.x;
  const tb::TreeSmem t = tb::tree_smem(smem, a);
  griddep_wait();
  griddep_launch_dependents();
  const bool bad = tb::stage_request(a, r, t, tid, kTreeThreads);
  const bool bad_cost = __syncthreads_or(bad) != 0;
  if (tid >= 32) return;  // warp 0 alone from here
  const int N = tb::pop_all<S>(a, t, tid);
  __syncwarp();
  tb::write_tree(a, r, t, N, bad_cost, tid, 32);
}

template <int S>
cudaError_t launch_s(const TreeArgs &a, size_t smem, cudaStream_t stream) {
  if (smem > 48 * 1024) {
    const cudaError_t e =
        cudaFuncSetAttribute(build_tree_kernel<S>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  return launch_pdl(build_tree_kernel<S>, dim3(a.B), dim3(kTreeThreads), smem, stream, a);
}

}  // namespace

int launch_build_tree(const float *topk_logit, const int32_t *topk_tok, const double *lse, int B,
                      int b, int K, int n_max, const int32_t *root_token, const int32_t *ctx_len,
                      const float *cost_ms, int cost_per_request, const float *l_ar,
                      int32_t *n_nodes, int32_t *parent, int32_t *depth, int32_t *pos_id,
                      int32_t *token, int32_t *rank, float *log_rho, float *a_hat, float *speedup,
                      uint32_t *anc_mask, int32_t *status, cudaStream_t stream) {
  const TreeArgs a = tb::tree_args(topk_logit, topk_tok, lse, B, b, K, n_max, root_token, ctx_len,
                                   cost_ms, cost_per_request, l_ar, n_nodes, parent, depth, pos_id,
                                   token, rank, log_rho, a_hat, speedup, anc_mask, status);
  const size_t smem = tb::tree_smem_bytes(b, a.R, n_max, a.W);
  cudaError_t e;
  switch (tb::tree_slots(n_max)) {
    case 1: e = launch_s<1>(a, smem, stream); break;
    case 2: e = launch_s<2>(a, smem, stream); break;
    case 4: e = launch_s<4>(a, smem, stream); break;
    default: e = launch_s<8>(a, smem, stream); break;
  }
  return (e == cudaSuccess && cudaGetLastError() == cudaSuccess) ? BASTION_OK : BASTION_ERR_LAUNCH;
}

}  // namespace bastion
