// Backward entry point for callers that cannot allocate device memory.
//
// Some callers of this library cannot call cudaMalloc: a host program that
// owns no device allocator of its own, a runtime whose device memory pool is
// sized once at start-up and forbids new allocations afterwards, or a hot loop
// where an allocation (which can synchronise the device and fragment memory)
// is not acceptable.  sinkattn_bwd needs a caller-provided workspace; this
// variant instead uses a fixed workspace compiled into the library as a
// file-scope device array, so the caller passes only inputs and outputs.
//
// Limits and rules:
//   * The array holds kStaticWorkspaceBytes (32 MiB).  A problem whose
//     sinkattn_bwd_workspace_size() exceeds that is rejected with
//     SINKATTN_ERR_WORKSPACE before anything is launched.
//   * Every GPU that loads the library holds the array until the process ends.
//   * The device address of the array is looked up once per device, on the
//     first call made while that device is current (cudaGetSymbolAddress).
//     Make that first call before any stream capture.
//   * All calls share the one array, and it keeps whatever the last call left
//     there.  Nothing in it has to start at zero: the backward preprocess
//     kernel clears the fp32 dQ accumulator before the main kernel adds into
//     it, and every other part (the per-row bias terms, the dsink partial
//     sums, the per-chunk dK/dV partial sums of split key tiles) is written
//     in full before it is read.  Calls whose kernels overlap on the GPU
//     (different streams, or several host threads) race on the array and give
//     wrong results: serialise them.
#include <mutex>

#include "../../include/sinkattn.h"
#include "internal.h"

namespace {

constexpr size_t kStaticWorkspaceBytes = size_t(32) << 20;
constexpr int kMaxDevices = 256;

static __device__ __align__(256) unsigned char g_static_workspace[kStaticWorkspaceBytes];

std::mutex g_setup_mutex;
void* g_workspace_ptr[kMaxDevices] = {};

// Device address of g_static_workspace for the current device (set up once).
sinkattn_status static_workspace(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SINKATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_workspace_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess || p == nullptr) return SINKATTN_ERR_CUDA;
    g_workspace_ptr[dev] = p;
  }
  *out = g_workspace_ptr[dev];
  return SINKATTN_OK;
}

}  // namespace

extern "C" sinkattn_status sinkattn_bwd_noalloc(const sinkattn_problem* prob, const void* q, const void* k,
                                                const void* v, const void* o, const float* lse, const void* dout,
                                                const float* sink, void* dq, void* dk, void* dv, float* dsink,
                                                void* stream) {
  const size_t need = sinkattn_bwd_workspace_size(prob);
  if (need == 0) {
    // Invalid problem: let the regular entry point report which check failed.
    return sinkattn_bwd(prob, q, k, v, o, lse, dout, sink, dq, dk, dv, dsink, nullptr, 0, stream);
  }
  if (need > kStaticWorkspaceBytes) return SINKATTN_ERR_WORKSPACE;
  void* ws = nullptr;
  const sinkattn_status st = static_workspace(&ws);
  if (st != SINKATTN_OK) return st;
  return sinkattn_bwd(prob, q, k, v, o, lse, dout, sink, dq, dk, dv, dsink, ws, kStaticWorkspaceBytes, stream);
}
