// Per-device runtime of the library: the device status word, per-device
// set-up (architecture check, SM count, the tensor-map encoder), launch
// counting and event timing behind ns_profile_*, the GEMM tiling override,
// and the bf16 tensor maps of the GEMM kernels.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>
#include <vector>

#include "orchestrate.h"
#include "status.h"

// Device status word (one per device context): kernels atomicOr NS_DEV_* bits.
__device__ unsigned int g_ns_status;

namespace nsorch {
namespace {

std::mutex g_mu;
unsigned int* g_status_ptr[nsplan::kMaxDevices] = {nullptr};
int g_sm_count[nsplan::kMaxDevices] = {0};
int g_cc_ok[nsplan::kMaxDevices] = {0};  // 0 unknown, 1 sm_103, -1 other

// set once under g_mu, read without it by every launch's tensor-map encoding
std::atomic<EncodeTiledFn> g_encode{nullptr};
int g_force_cl = 0;  // 0: automatic; otherwise the tiling mode of pick_cl
// test support: wait limit (ns) of the next bf16 GEMM launch, which then
// stalls (0: none armed)
std::atomic<unsigned long long> g_stall_next{0};
std::atomic<int> g_small_path{1};  // small buckets: one CTA per matrix
std::atomic<int> g_sym_mirror{0};  // bf16 A and B: 0 upper pair blocks only, 1 also the mirror

// ----------------------------------------------------------- measurement
std::mutex g_prof_mu;
bool g_prof_on = false;
long long g_launches[kKinds] = {0};
double g_ms[kKinds] = {0};
struct PendingTiming {
  cudaEvent_t a, b;
  int kind;
};
std::vector<PendingTiming> g_pending;
std::vector<cudaEvent_t> g_free_events;

cudaEvent_t take_event() {
  if (!g_free_events.empty()) {
    cudaEvent_t e = g_free_events.back();
    g_free_events.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

}  // namespace

bool prof_begin(int kind, cudaEvent_t* a, cudaEvent_t* b) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  ++g_launches[kind];
  if (g_prof_on) {
    *a = take_event();
    *b = take_event();
  }
  return g_prof_on;
}

void prof_end(int kind, cudaEvent_t a, cudaEvent_t b) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_pending.push_back({a, b, kind});
}

unsigned long long take_gemm_stall() { return g_stall_next.exchange(0); }

bool small_path_enabled() { return g_small_path.load() != 0; }

bool symmetric_mirror() { return g_sym_mirror.load() != 0; }

int gemm_cluster_override() {
  std::lock_guard<std::mutex> lk(g_mu);
  return g_force_cl;
}

EncodeTiledFn tensor_map_encoder() { return g_encode.load(std::memory_order_acquire); }

// Per-device set-up: status word address, SM count, architecture check.
int device_setup(int* dev_out, unsigned int** status_out, int* nsm_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return NS_ERR_CUDA;
  if (dev < 0 || dev >= nsplan::kMaxDevices) return NS_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_cc_ok[dev] == 0) {
    int major = 0, minor = 0, nsm = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return NS_ERR_CUDA;
    if (major != 10 || minor != 3) {
      g_cc_ok[dev] = -1;
      return NS_ERR_UNSUPPORTED;
    }
    void* sp = nullptr;
    if (cudaGetSymbolAddress(&sp, g_ns_status) != cudaSuccess) return NS_ERR_CUDA;
    g_status_ptr[dev] = static_cast<unsigned int*>(sp);
    g_sm_count[dev] = nsm;
    g_cc_ok[dev] = 1;
  }
  if (g_cc_ok[dev] < 0) return NS_ERR_UNSUPPORTED;
  if (!g_encode.load(std::memory_order_relaxed)) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return NS_ERR_CUDA;
    g_encode.store(reinterpret_cast<EncodeTiledFn>(fn), std::memory_order_release);
  }
  *dev_out = dev;
  *status_out = g_status_ptr[dev];
  *nsm_out = g_sm_count[dev];
  return NS_OK;
}

int make_map(CUtensorMap* m, void* base, uint64_t inner, uint64_t outer, uint64_t count, uint32_t box_inner,
             uint32_t box_outer, CUtensorMapSwizzle swz) {
  cuuint64_t dims[3] = {inner, outer, count};
  cuuint64_t strides[2] = {inner * 2, inner * outer * 2};
  cuuint32_t box[3] = {box_inner, box_outer, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = tensor_map_encoder()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? NS_OK : NS_ERR_CUDA;
}

int make_epi_map(CUtensorMap* m, void* base, uint64_t inner, uint64_t outer, uint64_t count) {
  return make_map(m, base, inner, outer, count, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
}

}  // namespace nsorch

using namespace nsorch;

extern "C" {

int ns_check_status(ns_plan_t* /*plan*/, void* stream) {
  int dev;
  unsigned int* status;
  int nsm;
  int rc = device_setup(&dev, &status, &nsm);
  if (rc != NS_OK) return rc;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return NS_ERR_CUDA;
  unsigned int word = 0;
  if (cudaMemcpy(&word, status, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return NS_ERR_CUDA;
  if (word) {
    const unsigned int zero = 0;
    if (cudaMemcpy(status, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return NS_ERR_CUDA;
    if (word & NS_DEV_TIMEOUT) return NS_ERR_TIMEOUT;
    return NS_ERR_DEVICE_CHECK;
  }
  if (cudaGetLastError() != cudaSuccess) return NS_ERR_CUDA;
  return NS_OK;
}

int ns_set_gemm_cluster(int cl) {
  if (cl != 0 && cl != 1 && cl != 3) return NS_ERR_ARG;
  std::lock_guard<std::mutex> lk(g_mu);
  g_force_cl = cl;
  return NS_OK;
}

int ns_set_small_path(int enable) {
  if (enable != 0 && enable != 1) return NS_ERR_ARG;
  g_small_path.store(enable);
  return NS_OK;
}

int ns_set_symmetric_store(int mode) {
  if (mode != 0 && mode != 1) return NS_ERR_ARG;
  g_sym_mirror.store(mode);
  return NS_OK;
}

int ns_test_stall_next_gemm(uint64_t wait_limit_ns) {
  if (wait_limit_ns < 100000ull || wait_limit_ns > 10000000000ull) return NS_ERR_ARG;
  g_stall_next.store(wait_limit_ns);
  return NS_OK;
}

int ns_profile_enable(int enable) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_prof_on = enable != 0;
  return NS_OK;
}

int ns_profile_read(int reset, int64_t* launches, double* gpu_ms) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  int rc = NS_OK;
  for (const PendingTiming& t : g_pending) {
    float ms = 0.0f;
    if (cudaEventSynchronize(t.b) != cudaSuccess || cudaEventElapsedTime(&ms, t.a, t.b) != cudaSuccess)
      rc = NS_ERR_CUDA;
    else
      g_ms[t.kind] += ms;
    g_free_events.push_back(t.a);
    g_free_events.push_back(t.b);
  }
  g_pending.clear();
  for (int k = 0; k < kKinds; ++k) {
    if (launches) launches[k] = g_launches[k];
    if (gpu_ms) gpu_ms[k] = g_ms[k];
    if (reset) {
      g_launches[k] = 0;
      g_ms[k] = 0.0;
    }
  }
  return rc;
}

}  // extern "C"
