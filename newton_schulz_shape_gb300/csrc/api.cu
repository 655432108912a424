// Device-side C ABI: ns_orthogonalize_batched, the shape-batched
// Newton-Schulz entry point (Megatron-Core API page owner_planning, ns_cost_fn:
// view, normalise, transpose so rows <= cols, then per step A = X X^T;
// X = a X + (b A + c A A) X; Megatron-LM issue #6720: NS batched by shape).
// It dispatches on the plan's precision policy to the bf16 or fp32
// orchestration. Nothing here allocates device memory; all per-call data
// travels in kernel parameter blocks.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <mutex>
#include <vector>

#include "orchestrate.h"
#include "status.h"

using namespace nsorch;

extern "C" {

int ns_orthogonalize_batched(ns_plan_t* plan, const void* const* in, void* const* out, int n, void* workspace,
                             uint64_t workspace_bytes, void* stream) {
  if (!plan) return NS_ERR_ARG;
  Plan& p = plan->p;
  if (n != static_cast<int>(p.part.size())) return NS_ERR_ARG;
  if (n == 0) return NS_OK;
  if (!in || !out) return NS_ERR_ARG;
  for (int j = 0; j < n; ++j) {
    const Tensor& t = p.t[p.part[j]];
    if (t.numel > 0 && (!in[j] || !out[j])) return NS_ERR_ARG;
  }
  if (p.buckets.empty()) return NS_OK;
  if (!workspace || workspace_bytes < p.ws_bytes || (reinterpret_cast<uintptr_t>(workspace) & 255))
    return NS_ERR_WORKSPACE;
  int dev;
  unsigned int* status;
  int nsm;
  int rc = device_setup(&dev, &status, &nsm);
  if (rc != NS_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  if (p.gram_mode == NS_FP32_GRAM) return orthogonalize_f32(p, in, out, ws, nsm, status, st);
  if (p.gram_mode == NS_FP32_GRAM_SPACE) return orthogonalize_gram_space(p, in, out, ws, nsm, status, st);
  if (p.gram_mode == NS_FP32_AUTO) {
    // per bucket: standard fp32-Gram iteration or Gram space, one workspace
    if (!plan->view_std.buckets.empty()) {
      rc = orthogonalize_f32(plan->view_std, in, out, ws, nsm, status, st);
      if (rc != NS_OK) return rc;
    }
    if (!plan->view_gs.buckets.empty()) return orthogonalize_gram_space(plan->view_gs, in, out, ws, nsm, status, st);
    return NS_OK;
  }

  rc = prologue_bf16(p, in, out, ws, status, st);
  if (rc != NS_OK) return rc;
  rc = small_bf16(p, in, out, status, st);
  if (rc != NS_OK) return rc;
  return steps_bf16(p, out, ws, nsm, status, st);
}

}  // extern "C"
