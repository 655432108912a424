// Routing between the S rank buffers and the S home buffers over one GPU's
// memory (Megatron-Core API page layer_sharded_a2a: route_to_ns_home /
// route_from_ns_home; page owner_planning: OwnerGatherPlan / OwnerScatterPlan):
// the plan's routing table, uploaded once per device, drives ns_pack_kernel.
// Also plan destruction, which frees those tables.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <mutex>
#include <vector>

#include "orchestrate.h"
#include "status.h"

namespace nsorch {
namespace {

// guards the lazily uploaded routing tables of all plans
std::mutex g_route_mu;

int upload_route(Plan& p, int dev) {
  if (p.d_route[dev] || p.route.empty()) return NS_OK;
  const size_t bytes = p.route.size() * sizeof(nsk::RouteEntry);
  void* d = nullptr;
  if (cudaMalloc(&d, bytes) != cudaSuccess) return NS_ERR_CUDA;
  if (cudaMemcpy(d, p.route.data(), bytes, cudaMemcpyHostToDevice) != cudaSuccess) {
    cudaFree(d);
    return NS_ERR_CUDA;
  }
  p.d_route[dev] = d;
  return NS_OK;
}

}  // namespace

int route(ns_plan_t* plan, void* const* rank_bufs, void* const* home_bufs, int S, int shard_dim, bool to_home,
          int elem_bytes, cudaStream_t st, long long g_begin, long long g_end) {
  if (!plan) return NS_ERR_ARG;
  Plan& p = plan->p;
  if (S != p.S) return NS_ERR_ARG;
  if (p.layout == NS_LAYOUT_ROW_SHARD ? shard_dim != p.shard_dim : shard_dim != 0) return NS_ERR_ARG;
  if (p.route.empty() || p.rank_len == 0) return NS_OK;
  if (!rank_bufs || !home_bufs) return NS_ERR_ARG;
  for (int r = 0; r < S; ++r) {
    if (!rank_bufs[r] && p.rank_len > 0) return NS_ERR_ARG;
    if (!home_bufs[r] && p.home_sizes[r] > 0) return NS_ERR_ARG;
  }
  int dev;
  unsigned int* status;
  int nsm;
  int rc = device_setup(&dev, &status, &nsm);
  if (rc != NS_OK) return rc;
  {
    std::lock_guard<std::mutex> lk(g_route_mu);
    rc = upload_route(p, dev);
  }
  if (rc != NS_OK) return rc;
  nsk::PackParams pp;
  std::memset(&pp, 0, sizeof(pp));
  for (int r = 0; r < S; ++r) {
    pp.rank_ptr[r] = rank_bufs[r];
    pp.home_ptr[r] = home_bufs[r];
  }
  pp.entries = static_cast<const nsk::RouteEntry*>(p.d_route[dev]);
  pp.n_entries = static_cast<long long>(p.route.size());
  pp.rank_len = p.rank_len;
  pp.chunk = 32768;
  pp.g_begin = g_begin;
  pp.g_end = g_end >= 0 ? g_end : (p.layout == NS_LAYOUT_FLAT ? p.rank_len * S : p.rank_len);
  pp.S = S;
  pp.T = p.layout == NS_LAYOUT_TWO_STAGE ? p.T : 1;
  pp.flat = p.layout == NS_LAYOUT_FLAT ? 1 : 0;
  pp.elem_bytes = elem_bytes;
  pp.to_home = to_home ? 1 : 0;
  pp.status = status;
  return counted(K_PACK, st, [&] { return nsk::launch_pack(pp, st); }) == cudaSuccess ? NS_OK : NS_ERR_CUDA;
}

}  // namespace nsorch

using namespace nsorch;

extern "C" {

int ns_pack_to_home(ns_plan_t* plan, const void* const* rank_bufs, int S, int shard_dim, void* const* home_bufs,
                    void* stream) {
  return route(plan, const_cast<void* const*>(rank_bufs), home_bufs, S, shard_dim, true,
               plan ? plan->p.in_bytes : 2, static_cast<cudaStream_t>(stream));
}

int ns_unpack_from_home(ns_plan_t* plan, const void* const* home_bufs, int S, int shard_dim, void* const* rank_bufs,
                        void* stream) {
  return route(plan, rank_bufs, const_cast<void* const*>(home_bufs), S, shard_dim, false,
               plan ? plan->p.out_bytes : 2, static_cast<cudaStream_t>(stream));
}

int ns_test_set_route_home(ns_plan_t* plan, int tensor, int home) {
  if (!plan || tensor < 0 || tensor >= static_cast<int>(plan->p.t.size())) return NS_ERR_ARG;
  Plan& p = plan->p;
  // the table holds one entry per participating tensor with data, in index order
  size_t k = 0;
  bool found = false;
  for (int i : p.part) {
    const Tensor& t = p.t[i];
    if (p.layout != NS_LAYOUT_FLAT ? t.shard_len == 0 : t.numel == 0) continue;
    if (i == tensor) {
      found = true;
      break;
    }
    ++k;
  }
  if (!found || k >= p.route.size()) return NS_ERR_ARG;
  std::lock_guard<std::mutex> lk(g_route_mu);
  p.route[k].home = home;
  int cur = 0;
  if (cudaGetDevice(&cur) != cudaSuccess) cur = -1;
  int rc = NS_OK;
  for (int d = 0; d < nsplan::kMaxDevices; ++d) {
    if (!p.d_route[d]) continue;
    nsk::RouteEntry* dev_e = static_cast<nsk::RouteEntry*>(p.d_route[d]) + k;
    if (cudaSetDevice(d) != cudaSuccess || cudaMemcpy(&dev_e->home, &home, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
      rc = NS_ERR_CUDA;
  }
  if (cur >= 0) cudaSetDevice(cur);
  return rc;
}

int ns_plan_destroy(ns_plan_t* plan) {
  if (!plan) return NS_OK;
  bool any = false;
  for (int d = 0; d < nsplan::kMaxDevices; ++d) any = any || plan->p.d_route[d] != nullptr;
  if (!any) {
    delete plan;
    return NS_OK;
  }
  int cur = -1;
  const bool have_dev = cudaGetDevice(&cur) == cudaSuccess;
  for (int d = 0; d < nsplan::kMaxDevices; ++d) {
    if (!plan->p.d_route[d]) continue;
    if (cudaSetDevice(d) == cudaSuccess) cudaFree(plan->p.d_route[d]);
    plan->p.d_route[d] = nullptr;
  }
  if (have_dev) cudaSetDevice(cur);
  delete plan;
  return NS_OK;
}

}  // extern "C"
