// Newton-Schulz without a caller-supplied workspace.
//
// ns_orthogonalize_batched needs scratch device memory (the two X buffers,
// A, B and the norm partial sums), which its caller allocates. Some callers
// cannot allocate device memory when they need this call: a plugin loaded into
// a host program whose caching allocator already owns the GPU's memory, or
// code that is not allowed to call cudaMalloc after start-up because an
// allocation may synchronise the device or fail under memory pressure. For
// them, ns_orthogonalize_batched_fixed_ws runs the same kernels on a scratch
// array that lives in this file as a static device array of fixed size.
//
// The array exists once per GPU that loads this library and is held until the
// process exits. It keeps the last call's contents; nothing needs clearing
// between calls, because every byte the kernels read is written earlier in
// the same call (the prologue writes X_0 including its zero padding, the Gram
// and A*A phases write every element of A and B, the B*X phase every element
// of the next X). All calls share the one array, so calls that overlap on the
// GPU (for example on two streams) race and give wrong results.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/nsgb300.h"
#include "plan.h"

namespace {

static __device__ __align__(256) unsigned char g_ns_fixed_ws[NS_FIXED_WS_BYTES];

std::mutex g_fixed_mu;
void* g_fixed_ptr[nsplan::kMaxDevices] = {nullptr};

// Device address of the array on the current device. In host code the
// array's name is only a host-side stand-in, so the address must come from
// cudaGetSymbolAddress, once per device, with that device current.
int fixed_ws_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return NS_ERR_CUDA;
  if (dev < 0 || dev >= nsplan::kMaxDevices) return NS_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_fixed_mu);
  if (!g_fixed_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_ns_fixed_ws) != cudaSuccess || !p) return NS_ERR_CUDA;
    g_fixed_ptr[dev] = p;
  }
  *out = g_fixed_ptr[dev];
  return NS_OK;
}

}  // namespace

extern "C" int ns_orthogonalize_batched_fixed_ws(ns_plan_t* plan, const void* const* in, void* const* out, int n,
                                                 void* stream) {
  if (!plan) return NS_ERR_ARG;
  uint64_t need = 0;
  int rc = ns_plan_workspace_bytes(plan, &need);
  if (rc != NS_OK) return rc;
  if (need > NS_FIXED_WS_BYTES) return NS_ERR_WORKSPACE;
  if (need == 0) return ns_orthogonalize_batched(plan, in, out, n, nullptr, 0, stream);
  void* ws = nullptr;
  rc = fixed_ws_address(&ws);
  if (rc != NS_OK) return rc;
  return ns_orthogonalize_batched(plan, in, out, n, ws, NS_FIXED_WS_BYTES, stream);
}
