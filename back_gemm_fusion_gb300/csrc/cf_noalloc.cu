// cf_noalloc.cu -- cf_gemm_epilogue_noalloc: the fused GEMM + epilogue call
// for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocator) at the point where
// they run the fused kernel: code that must have bounded latency (cudaMalloc
// may synchronise the device), plugins whose host framework owns every
// allocation and hands out no allocator, and code paths that must not
// allocate in steady state.  For rows wider than one CTA tile the fused
// kernel needs a small scratch area (per-tile partial row statistics and
// arrival counters).  This entry point takes that scratch from a file-scope
// device array instead of a caller-provided workspace, so it allocates
// nothing.  The caller still passes the inputs and the output.
//
// Limits and sharing:
//   * The array holds CF_NOALLOC_WORKSPACE_BYTES bytes.  It is part of the
//     loaded library, so every GPU that loads the library holds it until the
//     process exits.  Problems whose scratch would exceed it are rejected with
//     CF_ERR_WORKSPACE before anything is enqueued.
//   * Every call shares the one array, which keeps the previous call's
//     contents; the call clears the arrival counters (the part that must
//     start at zero) on the caller's stream before the kernel runs.  Calls
//     whose executions overlap on the GPU (different streams, or several
//     host threads) race on the array: serialise them.
//   * The first call on a device looks up the array's device address with
//     cudaGetSymbolAddress on that device (the device must be current).  Make
//     that first call before any stream capture.
#include <cuda_runtime.h>

#include <mutex>

#include "cf_internal.h"

// The scratch array.  In host code this name is only a host-side stand-in:
// its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_cf_noalloc_ws[CF_NOALLOC_WORKSPACE_BYTES];

namespace {
constexpr int kMaxDev = 64;
std::mutex g_mu;
void* g_addr[kMaxDev] = {};

// Device address of the scratch array on the current device (set up once).
cf_status scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
    cudaGetLastError();
    return CF_ERR_NO_DEVICE;
  }
  if (dev >= kMaxDev) return CF_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_cf_noalloc_ws);
    if (e != cudaSuccess || !p) {
      cudaGetLastError();
      return CF_ERR_CUDA;
    }
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return CF_OK;
}
}  // namespace

extern "C" cf_status cf_gemm_epilogue_noalloc(const cf_matrix* A, const cf_matrix* B, const float* bias,
                                              const float* gamma, const float* beta, const cf_epi_desc* epi,
                                              cf_matrix* out, void* stream) {
  // Host-only size check first: nothing is enqueued for oversized problems.
  const size_t need = cf_workspace_size(A, B, epi);
  if (need > (size_t)CF_NOALLOC_WORKSPACE_BYTES) return CF_ERR_WORKSPACE;
  void* ws = nullptr;
  if (need > 0) {
    const cf_status s = scratch_address(&ws);
    if (s != CF_OK) return s;
  }
  return cf_gemm_epilogue(A, B, bias, gamma, beta, epi, out, ws, need > 0 ? (size_t)CF_NOALLOC_WORKSPACE_BYTES : 0,
                          stream);
}
