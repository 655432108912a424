// Wave pipeline (ns_pipeline_*): Megatron-LM issue #6720 wave dispatch in a
// single-GPU form.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <mutex>
#include <vector>

#include "orchestrate.h"
#include "status.h"

using namespace nsorch;

namespace {

// ------------------------------------------------------------ wave pipeline
// Megatron-LM issue #6720: NS work statically partitioned into waves that are
// dispatched as their inputs become ready, so the exchange of one wave hides
// behind the NS of another. Single-GPU form: W waves of consecutive tensors
// (cost-balanced), three streams -- memory (pack + prologue of wave w+1),
// GEMM (NS steps of wave w), out (unpack of wave w-1) -- and two workspace
// halves that alternate between waves.
struct PipeDev {
  cudaStream_t mem = nullptr, gemm = nullptr, out = nullptr;
  std::vector<cudaEvent_t> ev;  // start, end x3, then per wave: pro, gemm
};

}  // namespace

struct ns_pipeline {
  ns_plan_t* base = nullptr;
  int W = 0;
  std::vector<nsplan::Plan> wave;
  std::vector<long long> g_begin, g_end;
  uint64_t ws_half = 0;
  PipeDev dev[nsplan::kMaxDevices];
};

namespace {

void release(PipeDev& pd) {
  for (cudaEvent_t e : pd.ev)
    if (e) cudaEventDestroy(e);
  pd.ev.clear();
  for (cudaStream_t* s : {&pd.mem, &pd.gemm, &pd.out}) {
    if (*s) cudaStreamDestroy(*s);
    *s = nullptr;
  }
}

// streams and events of one device, created on first use; all or nothing, so
// a failed set-up is retried by the next call
int pipe_device(ns_pipeline* pl, int d) {
  PipeDev& pd = pl->dev[d];
  if (pd.mem) return NS_OK;
  PipeDev nd;
  bool ok = cudaStreamCreateWithFlags(&nd.mem, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&nd.gemm, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&nd.out, cudaStreamNonBlocking) == cudaSuccess;
  if (ok) {
    nd.ev.assign(4 + 2 * pl->W, nullptr);
    for (cudaEvent_t& e : nd.ev) ok = ok && cudaEventCreateWithFlags(&e, cudaEventDisableTiming) == cudaSuccess;
  }
  if (!ok) {
    release(nd);
    return NS_ERR_CUDA;
  }
  pd = nd;
  return NS_OK;
}

}  // namespace

extern "C" {

int ns_pipeline_create(ns_plan_t* plan, int n_waves, ns_pipeline_t** out) {
  if (!out) return NS_ERR_ARG;
  *out = nullptr;
  if (!plan || n_waves < 1) return NS_ERR_ARG;
  const Plan& p = plan->p;
  if (p.gram_mode != NS_BF16) return NS_ERR_UNSUPPORTED;
  const int np = static_cast<int>(p.part.size());
  ns_pipeline* pl = new (std::nothrow) ns_pipeline();
  if (!pl) return NS_ERR_ARG;
  pl->base = plan;
  if (np == 0) {
    // nothing participates: no waves, and a run only orders the streams
    *out = pl;
    return NS_OK;
  }
  // Waves overlap one wave's prologue with the previous wave's GEMMs. When
  // every bucket runs as one CTA per matrix there is nothing to overlap, and a
  // split would only add launches: one wave then.
  bool all_small = small_path_enabled();
  for (const nsplan::Bucket& b : p.buckets) all_small = all_small && b.small;
  const int W = all_small ? 1 : std::min(n_waves, np);
  // cost-balanced cut of the participating tensors (index order) into W waves
  double total = 0;
  for (int i : p.part) total += static_cast<double>(std::max<int64_t>(p.t[i].cost, 1));
  std::vector<std::vector<int>> members(1);
  double acc = 0;
  for (int k = 0; k < np; ++k) {
    const int i = p.part[k];
    const int left_tensors = np - k;
    const int left_waves = W - static_cast<int>(members.size());
    if (!members.back().empty() && left_waves > 0 &&
        (acc >= total * members.size() / W || left_tensors <= left_waves))
      members.emplace_back();
    members.back().push_back(i);
    acc += static_cast<double>(std::max<int64_t>(p.t[i].cost, 1));
  }
  pl->W = static_cast<int>(members.size());
  pl->wave.resize(pl->W);
  for (int w = 0; w < pl->W; ++w) {
    int rc = nsplan::build_subplan(p, members[w], pl->wave[w]);
    if (rc != NS_OK) {
      delete pl;
      return rc;
    }
    const Tensor& f = p.t[members[w].front()];
    const Tensor& l = p.t[members[w].back()];
    if (p.layout == NS_LAYOUT_FLAT) {
      pl->g_begin.push_back(f.flat_off);
      pl->g_end.push_back(l.flat_off + l.numel);
    } else {
      pl->g_begin.push_back(f.rank_off);
      pl->g_end.push_back(l.rank_off + l.shard_len);
    }
    pl->ws_half = std::max(pl->ws_half, (pl->wave[w].ws_bytes + 1023) / 1024 * 1024);
  }
  *out = pl;
  return NS_OK;
}

int ns_pipeline_info(const ns_pipeline_t* pl, int* n_waves, uint64_t* workspace_bytes) {
  if (!pl) return NS_ERR_ARG;
  if (n_waves) *n_waves = pl->W;
  if (workspace_bytes) *workspace_bytes = 2 * pl->ws_half;
  return NS_OK;
}

int ns_pipeline_run(ns_pipeline_t* pl, const void* const* rank_in, void* const* home_in, void* const* home_out,
                    void* const* rank_out, void* workspace, uint64_t workspace_bytes, void* stream) {
  if (!pl || !pl->base) return NS_ERR_ARG;
  Plan& p = pl->base->p;
  const int S = p.S;
  if (!rank_in || !home_in || !home_out || !rank_out) return NS_ERR_ARG;
  if (pl->ws_half > 0 &&
      (!workspace || workspace_bytes < 2 * pl->ws_half || (reinterpret_cast<uintptr_t>(workspace) & 255)))
    return NS_ERR_WORKSPACE;
  int dev;
  unsigned int* status;
  int nsm;
  int rc = device_setup(&dev, &status, &nsm);
  if (rc != NS_OK) return rc;
  rc = pipe_device(pl, dev);
  if (rc != NS_OK) return rc;
  PipeDev& pd = pl->dev[dev];
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaEvent_t* ev = pd.ev.data();
  const int sd = p.layout == NS_LAYOUT_ROW_SHARD ? p.shard_dim : 0;
  // row shards along dim 0: every row of a tensor is contiguous in one rank
  // buffer, so the prologue reads the rank buffers and the pack to home_in is
  // skipped
  const bool fused_pack = p.layout == NS_LAYOUT_ROW_SHARD && p.shard_dim == 0;
  if (pl->W == 1 && fused_pack && !pl->wave[0].buckets.empty() && gemm_buckets(pl->wave[0]) == 0) {
    // every bucket runs as one CTA per matrix reading and writing the rank
    // buffers: the whole call is one launch, issued on the caller's stream
    // (nothing to overlap, so no fork onto the pipeline's streams and no join)
    const Plan& wp = pl->wave[0];
    std::vector<const void*> ins(wp.part.size(), nullptr);
    std::vector<void*> outs(wp.part.size(), nullptr);
    return small_bf16(wp, ins.data(), outs.data(), status, st, rank_in, rank_out);
  }
  if (cudaEventRecord(ev[0], st) != cudaSuccess || cudaStreamWaitEvent(pd.mem, ev[0], 0) != cudaSuccess ||
      cudaStreamWaitEvent(pd.gemm, ev[0], 0) != cudaSuccess || cudaStreamWaitEvent(pd.out, ev[0], 0) != cudaSuccess)
    return NS_ERR_CUDA;
  std::vector<const void*> ins;
  std::vector<void*> outs;
  for (int w = 0; w < pl->W; ++w) {
    const Plan& wp = pl->wave[w];
    char* ws = static_cast<char*>(workspace) + (w % 2) * pl->ws_half;
    cudaEvent_t ev_pro = ev[4 + 2 * w], ev_gemm = ev[5 + 2 * w];
    if (w >= 2 && cudaStreamWaitEvent(pd.mem, ev[5 + 2 * (w - 2)], 0) != cudaSuccess) return NS_ERR_CUDA;
    if (!fused_pack) {
      rc = route(pl->base, const_cast<void* const*>(rank_in), home_in, S, sd, true, p.in_bytes, pd.mem,
                 pl->g_begin[w], pl->g_end[w]);
      if (rc != NS_OK) return rc;
    }
    ins.assign(wp.part.size(), nullptr);
    outs.assign(wp.part.size(), nullptr);
    for (size_t j = 0; j < wp.part.size(); ++j) {
      const Tensor& t = wp.t[wp.part[j]];
      ins[j] = static_cast<const char*>(home_in[t.home]) + t.home_off * p.in_bytes;
      outs[j] = static_cast<char*>(home_out[t.home]) + t.home_off * p.out_bytes;
    }
    if (!wp.buckets.empty()) {
      rc = prologue_bf16(wp, ins.data(), outs.data(), ws, status, pd.mem, fused_pack ? rank_in : nullptr);
      if (rc != NS_OK) return rc;
    }
    if (cudaEventRecord(ev_pro, pd.mem) != cudaSuccess || cudaStreamWaitEvent(pd.gemm, ev_pro, 0) != cudaSuccess)
      return NS_ERR_CUDA;
    // the last B*X launches write the rank buffers themselves when the pack
    // was fused and every launch can store its results
    const bool fused_unpack = fused_pack && !wp.buckets.empty() && final_stores_all(wp);
    if (!wp.buckets.empty()) {
      rc = small_bf16(wp, ins.data(), outs.data(), status, pd.gemm, fused_pack ? rank_in : nullptr,
                      fused_unpack ? rank_out : nullptr);
      if (rc != NS_OK) return rc;
      rc = steps_bf16(wp, outs.data(), ws, nsm, status, pd.gemm, fused_unpack ? rank_out : nullptr);
      if (rc != NS_OK) return rc;
    }
    if (cudaEventRecord(ev_gemm, pd.gemm) != cudaSuccess || cudaStreamWaitEvent(pd.out, ev_gemm, 0) != cudaSuccess)
      return NS_ERR_CUDA;
    if (!fused_unpack) {
      rc = route(pl->base, rank_out, const_cast<void* const*>(home_out), S, sd, false, p.out_bytes, pd.out,
                 pl->g_begin[w], pl->g_end[w]);
      if (rc != NS_OK) return rc;
    }
  }
  if (cudaEventRecord(ev[1], pd.mem) != cudaSuccess || cudaEventRecord(ev[2], pd.gemm) != cudaSuccess ||
      cudaEventRecord(ev[3], pd.out) != cudaSuccess || cudaStreamWaitEvent(st, ev[1], 0) != cudaSuccess ||
      cudaStreamWaitEvent(st, ev[2], 0) != cudaSuccess || cudaStreamWaitEvent(st, ev[3], 0) != cudaSuccess)
    return NS_ERR_CUDA;
  return NS_OK;
}

int ns_pipeline_destroy(ns_pipeline_t* pl) {
  if (!pl) return NS_OK;
  int cur = -1;
  bool any = false;
  for (int d = 0; d < nsplan::kMaxDevices; ++d) any = any || pl->dev[d].mem != nullptr;
  if (any) {
    const bool have = cudaGetDevice(&cur) == cudaSuccess;
    for (int d = 0; d < nsplan::kMaxDevices; ++d) {
      PipeDev& pd = pl->dev[d];
      if (!pd.mem) continue;
      if (cudaSetDevice(d) != cudaSuccess) continue;
      release(pd);
    }
    if (have) cudaSetDevice(cur);
  }
  delete pl;
  return NS_OK;
}

}  // extern "C"
