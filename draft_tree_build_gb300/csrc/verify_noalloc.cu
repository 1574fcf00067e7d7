// Greedy verification for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc or ask anyone else to allocate for them:
// a serving loop that must never touch the allocator after start-up (an
// allocation can synchronise the device or fail under memory pressure), code
// running inside a framework whose allocator it does not own, or a plug-in
// that only receives input and output pointers.  For them this file offers one
// more entry point, bastion_verify_greedy_noalloc, whose scratch lives in a
// fixed array compiled into the library instead of a caller-provided workspace.
//
// The array below is a file-scope __device__ array: every GPU that loads the
// library holds it (128 KiB) until the process exits.  Its name is only a
// host-side stand-in in host code, so the host looks up its device address
// once per device with cudaGetSymbolAddress (with that device current) and
// passes that address to the kernel.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "bastion.h"

namespace bastion {
size_t verify_workspace_bytes(int B, int n_max);
int launch_verify(const void *target, int dtype, int B, int n_max, int V, int64_t ld, int b,
                  const int32_t *n_nodes, const int32_t *parent, const int32_t *token,
                  int32_t *argmax, int32_t *accept_len, int32_t *accept_nodes,
                  int32_t *out_tokens, void *ws, int32_t *status, cudaStream_t stream);
}  // namespace bastion

namespace {

// Largest sizes the fixed scratch covers: B * n_max <= 16384 node rows (one
// 8-byte key each) and B <= 4096 requests.
constexpr int kMaxRows = 16384;
constexpr int kMaxRequests = 4096;
constexpr size_t kScratchBytes = (size_t)kMaxRows * 8;

static __device__ __align__(256) unsigned char g_verify_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once per
// device); nullptr if the lookup fails.
void *scratch_for_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_verify_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();  // consume the error: it must not be reported by a later call
      return nullptr;
    }
    g_scratch_addr[dev] = p;
  }
  return g_scratch_addr[dev];
}

}  // namespace

extern "C" int bastion_verify_greedy_noalloc(const void *target_logits, int dtype, int B,
                                             int n_max, int V, int64_t ld_row, int b,
                                             const int32_t *n_nodes, const int32_t *parent,
                                             const int32_t *token, int32_t *argmax,
                                             int32_t *accept_len, int32_t *accept_nodes,
                                             int32_t *out_tokens, int32_t *status,
                                             bastion_stream_t stream) {
  if (!target_logits || !n_nodes || !parent || !token || !argmax || !accept_len ||
      !accept_nodes || !out_tokens || !status)
    return BASTION_ERR_NULL;
  if (dtype != BASTION_F32 && dtype != BASTION_BF16) return BASTION_ERR_DTYPE;
  if (B < 1 || B > 4096 || n_max < 1 || n_max > 256 || V < 1 || V >= (1 << 30) || ld_row < V ||
      b < 1 || b > 32)
    return BASTION_ERR_SIZE;
  // beyond what the fixed scratch holds
  if (B > kMaxRequests || (long long)B * n_max > kMaxRows) return BASTION_ERR_SIZE;
  const int es = dtype == BASTION_F32 ? 4 : 2;
  if ((uintptr_t)target_logits % es) return BASTION_ERR_ALIGN;
  const size_t need = bastion::verify_workspace_bytes(B, n_max);
  if (need > kScratchBytes) return BASTION_ERR_SIZE;
  void *scratch = scratch_for_current_device();
  if (!scratch) return BASTION_ERR_LAUNCH;
  // The array keeps whatever the previous call left; the keys this call uses
  // must start at zero.
  if (cudaMemsetAsync(scratch, 0, need, (cudaStream_t)stream) != cudaSuccess) {
    cudaGetLastError();  // consume the error: it must not be reported by a later call
    return BASTION_ERR_LAUNCH;
  }
  return bastion::launch_verify(target_logits, dtype, B, n_max, V, ld_row, b, n_nodes, parent,
                                token, argmax, accept_len, accept_nodes, out_tokens, scratch,
                                status, (cudaStream_t)stream);
}
