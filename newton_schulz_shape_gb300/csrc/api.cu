// Device-side C ABI: shape-batched Newton-Schulz orchestration, pack/unpack,
// the device status word, and plan destruction.
//
// ns_orthogonalize_batched follows the Megatron-Core API page owner_planning
// (ns_cost_fn: view, normalise, transpose so rows <= cols, then per step
// A = X X^T; X = a X + (b A + c A A) X) and the Megatron-LM issue #6720
// (NS batched by shape, symmetric SYRK-style Gram kernels): tensors of equal (m, n)
// form a bucket laid out as one [count, m_pad, n_pad] array in the caller's
// workspace, and every phase of every step runs as one persistent launch over
// the tiles of all buckets. Nothing here allocates device memory; all
// per-call data travels in kernel parameter blocks.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/nsgb300.h"
#include "kernels.h"
#include "plan.h"
#include "status.h"

// Device status word (one per device context): kernels atomicOr NS_DEV_* bits.
__device__ unsigned int g_ns_status;

namespace {

using nsplan::Bucket;
using nsplan::Plan;
using nsplan::Tensor;

std::mutex g_mu;
unsigned int* g_status_ptr[nsplan::kMaxDevices] = {nullptr};
int g_sm_count[nsplan::kMaxDevices] = {0};
int g_cc_ok[nsplan::kMaxDevices] = {0};  // 0 unknown, 1 sm_103, -1 other

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
int g_force_cl = 0;  // 0: automatic; otherwise the tiling mode of pick_cl

// ----------------------------------------------------------- measurement
constexpr int kKinds = 6;
enum { K_GRAM = 0, K_A2B = 1, K_BX = 2, K_PRO = 3, K_PACK = 4, K_BX_FINAL = 5 };
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

// Launch through `fn`, counting it and, if timing is on, bracketing it with
// events on `st`.
template <typename F>
cudaError_t counted(int kind, cudaStream_t st, F&& fn) {
  bool timed;
  cudaEvent_t a = nullptr, b = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    ++g_launches[kind];
    timed = g_prof_on;
    if (timed) {
      a = take_event();
      b = take_event();
    }
  }
  if (timed && a) cudaEventRecord(a, st);
  cudaError_t e = fn();
  if (timed && b) {
    cudaEventRecord(b, st);
    std::lock_guard<std::mutex> lk(g_prof_mu);
    g_pending.push_back({a, b, kind});
  }
  return e;
}

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
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return NS_ERR_CUDA;
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  *dev_out = dev;
  *status_out = g_status_ptr[dev];
  *nsm_out = g_sm_count[dev];
  return NS_OK;
}

// 3-D bf16 tensor map over [count][outer][inner] with a {box_inner, box_outer, 1}
// box, 128-byte swizzle (operand tiles) or 64-byte swizzle (epilogue chunks of
// 32 x 32), zero fill outside the array.
int make_map(CUtensorMap* m, void* base, uint64_t inner, uint64_t outer, uint64_t count, uint32_t box_inner,
             uint32_t box_outer, CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
  cuuint64_t dims[3] = {inner, outer, count};
  cuuint64_t strides[2] = {inner * 2, inner * outer * 2};
  cuuint32_t box[3] = {box_inner, box_outer, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? NS_OK : NS_ERR_CUDA;
}

int make_epi_map(CUtensorMap* m, void* base, uint64_t inner, uint64_t outer, uint64_t count) {
  return make_map(m, base, inner, outer, count, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
}

// Upper-triangle work items of one matrix: single tiles (cl = 1) or pairs of
// tile rows 2q, 2q + 1 sharing their column tiles (cl = 2).
long long syrk_tiles(int tiles_m, int tiles_n, int cl = 1) {
  long long t = 0;
  if (cl == 1) {
    for (int tm = 0; tm < tiles_m; ++tm) t += tiles_n - (tm * nsk::GEMM_BM) / nsk::GEMM_BN;
  } else {
    for (int q = 0; q < (tiles_m + 1) / 2; ++q) t += tiles_n - q;
  }
  return t;
}

// GEMM tiling for a launch: 1 = one CTA per 128 x 256 tile; 2 = CTA pairs
// sharing B tiles by multicast; 3 = CTA pairs running the 2-SM MMA on
// 256 x 256 tiles. Pairs need every bucket of the launch to have at least two
// tile rows.
int pick_cl(const Plan& p, size_t b0, size_t b1, int phase) {
  for (size_t bi = b0; bi < b1; ++bi) {
    const Bucket& b = p.buckets[bi];
    if (b.m_pad / nsk::GEMM_BM < 2) return 1;
  }
  if (g_force_cl) return g_force_cl;
  // Measured (interleaved runs on one plan): the 2-SM MMA is faster for the
  // Gram (K = n) everywhere, and for A*A and B*X when every bucket has an even
  // number of tile rows (GPT-style and Llama-shaped: 16 and 32 rows); with an
  // odd count the spare half of the last pair makes the 1-SM kernel faster
  // for those two (MoE 1408-row experts: 11 rows).
  if (phase != nsk::PH_GRAM)
    for (size_t bi = b0; bi < b1; ++bi)
      if ((p.buckets[bi].m_pad / nsk::GEMM_BM) % 2) return 1;
  return 3;
}

// Work items per matrix count tile-row pairs for both paired modes.
int count_mode(int cl) { return cl == 1 ? 1 : 2; }

struct BucketPtrs {
  char* x0;
  char* x1;
  char* a;
  char* b;
  float* partial;
  float* scale;
};

BucketPtrs bucket_ptrs(const Bucket& b, char* ws) {
  BucketPtrs q;
  q.x0 = ws + b.off_x0;
  q.x1 = ws + b.off_x1;
  q.a = ws + b.off_a;
  q.b = ws + b.off_b;
  q.partial = reinterpret_cast<float*>(ws + b.off_partial);
  q.scale = reinterpret_cast<float*>(ws + b.off_scale);
  return q;
}

// Fill the launch parameters of `phase` for buckets [b0, b1). `cur_is_x0`
// selects the X buffer the step reads. With `final_out` (B*X phase of the
// last step), every matrix's result goes straight to out[ordinal]: the table
// entry is the output address with bit 0 set for transposed tensors.
template <typename P>
int fill_phase(P& gp, const Plan& p, char* ws, int phase, bool cur_is_x0, size_t b0, size_t b1,
               unsigned int* status, void* const* final_out, int cl, bool first_step,
               void* const* final_ranks = nullptr) {
  std::memset(&gp, 0, sizeof(gp));
  gp.alpha = p.a;
  gp.beta = p.b;
  gp.gamma = p.c;
  gp.status = status;
  long long tiles = 0;
  int nb = 0, n_out = 0;
  for (size_t bi = b0; bi < b1; ++bi, ++nb) {
    const Bucket& b = p.buckets[bi];
    const BucketPtrs q = bucket_ptrs(b, ws);
    char* cur = cur_is_x0 ? q.x0 : q.x1;
    char* nxt = cur_is_x0 ? q.x1 : q.x0;
    const uint64_t cnt = b.members.size();
    nsk::GemmBucket& g = gp.bk[nb];
    // output maps exist in the parameter blocks of launches that store by TMA
    CUtensorMap* tmo = sizeof(gp.tmo) / sizeof(gp.tmo[0]) > 1 ? &gp.tmo[nb] : nullptr;
    g.tile_begin = tiles;
    g.count = static_cast<int>(cnt);
    g.tiles_m = static_cast<int>(b.m_pad / nsk::GEMM_BM);
    g.m_valid = static_cast<int>(b.m);
    g.n_valid = static_cast<int>(b.n);
    // X~_0 is unscaled: the first step's Gram and B*X apply the scale
    g.scale = first_step && phase != nsk::PH_A2B ? q.scale : nullptr;
    int rc = NS_OK;
    if (phase == nsk::PH_GRAM || phase == nsk::PH_A2B) {
      g.tiles_n = static_cast<int>((b.m_pad + nsk::GEMM_BN - 1) / nsk::GEMM_BN);
      g.tiles_per_mat = static_cast<int>(syrk_tiles(g.tiles_m, g.tiles_n, cl));
      g.cols_valid = static_cast<int>(b.m_pad);
      g.ld_out = static_cast<int>(b.m_pad);
      g.out_stride = b.m_pad * b.m_pad;
      if (phase == nsk::PH_GRAM) {
        g.k_blocks = static_cast<int>(b.n_pad / nsk::GEMM_BK);
        g.out = q.a;
        g.aux = nullptr;
        rc = make_map(&gp.tma[nb], cur, b.n_pad, b.m_pad, cnt, 64, 128);
        if (rc == NS_OK) rc = make_map(&gp.tmb[nb], cur, b.n_pad, b.m_pad, cnt, 64, 128);
        if (rc == NS_OK) rc = tmo ? make_epi_map(tmo, q.a, b.m_pad, b.m_pad, cnt) : NS_ERR_UNSUPPORTED;
      } else {
        g.k_blocks = static_cast<int>(b.m_pad / nsk::GEMM_BK);
        g.out = q.b;
        g.aux = q.a;
        g.ld_aux = static_cast<int>(b.m_pad);
        g.aux_stride = b.m_pad * b.m_pad;
        rc = make_map(&gp.tma[nb], q.a, b.m_pad, b.m_pad, cnt, 64, 128);
        if (rc == NS_OK) rc = make_map(&gp.tmb[nb], q.a, b.m_pad, b.m_pad, cnt, 64, 128);
        if (rc == NS_OK) rc = make_epi_map(&gp.tme[nb], q.a, b.m_pad, b.m_pad, cnt);
        if (rc == NS_OK) rc = tmo ? make_epi_map(tmo, q.b, b.m_pad, b.m_pad, cnt) : NS_ERR_UNSUPPORTED;
      }
    } else {
      g.tiles_n = static_cast<int>((b.n_pad + nsk::GEMM_BN - 1) / nsk::GEMM_BN);
      g.tiles_per_mat = (cl == 1 ? g.tiles_m : (g.tiles_m + 1) / 2) * g.tiles_n;
      g.cols_valid = static_cast<int>(b.n_pad);
      g.k_blocks = static_cast<int>(b.m_pad / nsk::GEMM_BK);
      g.out = nxt;
      g.aux = cur;
      g.ld_out = static_cast<int>(b.n_pad);
      g.ld_aux = static_cast<int>(b.n_pad);
      g.out_stride = b.m_pad * b.n_pad;
      g.aux_stride = b.m_pad * b.n_pad;
      rc = make_map(&gp.tma[nb], q.b, b.m_pad, b.m_pad, cnt, 64, 128);
      if (rc == NS_OK) rc = make_map(&gp.tmb[nb], cur, b.n_pad, b.m_pad, cnt, 64, 64);
      if (rc == NS_OK) rc = make_epi_map(&gp.tme[nb], cur, b.n_pad, b.m_pad, cnt);
      if (rc == NS_OK && !final_out) rc = tmo ? make_epi_map(tmo, nxt, b.n_pad, b.m_pad, cnt) : NS_ERR_UNSUPPORTED;
      if (final_out) {
        g.out_first = n_out;
        for (size_t s = 0; s < cnt; ++s) {
          const Tensor& t = p.t[b.members[s]];
          // the tensor's output address, or (row shards along dim 0) its
          // shard offset in every rank buffer
          const unsigned long long a = final_ranks ? static_cast<unsigned long long>(t.rank_off) << 1
                                                   : reinterpret_cast<unsigned long long>(final_out[t.ordinal]);
          gp.out_tab[n_out++] = a | (t.transposed ? 1ull : 0ull);
        }
      }
    }
    if (rc != NS_OK) return rc;
    tiles += static_cast<long long>(g.tiles_per_mat) * static_cast<long long>(cnt);
  }
  gp.nb = nb;
  gp.total_tiles = tiles;
  if (final_ranks) {
    gp.out_ranks = 1;
    gp.S = p.S;
    for (int r = 0; r < p.S; ++r) gp.rank_ptr[r] = final_ranks[r];
  }
  return NS_OK;
}

int run_phase(const Plan& p, char* ws, int phase, bool cur_is_x0, size_t b0, size_t b1, int nsm,
              unsigned int* status, bool first_step, bool reverse, cudaStream_t st) {
  nsk::GemmParams gp;
  const int cl = pick_cl(p, b0, b1, phase);
  int rc = fill_phase(gp, p, ws, phase, cur_is_x0, b0, b1, status, nullptr, count_mode(cl), first_step);
  if (rc != NS_OK) return rc;
  gp.reverse = reverse ? 1 : 0;
  return counted(phase, st, [&] {
           return cl == 3 ? nsk::launch_gemm_pair(phase, gp, nsm, st) : nsk::launch_gemm(phase, cl, gp, nsm, st);
         }) == cudaSuccess
             ? NS_OK
             : NS_ERR_CUDA;
}

// B*X phase of the last step, storing results directly into `out`, or with
// rank_out (row shards along dim 0) into the S rank buffers.
int run_final_bx(const Plan& p, char* ws, bool cur_is_x0, size_t b0, size_t b1, int nsm, unsigned int* status,
                 void* const* out, bool first_step, bool reverse, cudaStream_t st, void* const* rank_out = nullptr) {
  static thread_local nsk::GemmFinalParams gp;  // ~32 KB: kept off the stack
  const int cl = pick_cl(p, b0, b1, nsk::PH_BX);
  int rc = fill_phase(gp, p, ws, nsk::PH_BX, cur_is_x0, b0, b1, status, out, count_mode(cl), first_step, rank_out);
  gp.reverse = reverse ? 1 : 0;
  if (rc != NS_OK) return rc;
  return counted(K_BX_FINAL, st, [&] {
           return cl == 3 ? nsk::launch_gemm_pair_final(gp, nsm, st) : nsk::launch_gemm_final(cl, gp, nsm, st);
         }) == cudaSuccess
             ? NS_OK
             : NS_ERR_CUDA;
}

size_t group_matrices(const Plan& p, size_t b0, size_t b1) {
  size_t n = 0;
  for (size_t bi = b0; bi < b1; ++bi) n += p.buckets[bi].members.size();
  return n;
}

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

// Pack (to_home) or unpack the entry-coordinate range [g_begin, g_end)
// (g_end < 0: everything).
int route(ns_plan_t* plan, void* const* rank_bufs, void* const* home_bufs, int S, int shard_dim, bool to_home,
          int elem_bytes, cudaStream_t st, long long g_begin = 0, long long g_end = -1) {
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
    std::lock_guard<std::mutex> lk(g_mu);
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

// ------------------------------------------------------ fp32-Gram path
// Workspace per bucket (fp32): X sets 0 and 1 = [X hi | X lo | X^T hi | X^T lo]
// of cnt * m_pad * n_pad each; A = [hi | lo], B = [hi | lo] of cnt * m_pad^2.
struct Bucket32Ptrs {
  float* x[2];   // set base (X hi); X lo, X^T hi, X^T lo follow at xs apart
  float* a;      // A hi; A lo at as apart
  float* b;
  long long xs, as;
};

Bucket32Ptrs bucket32_ptrs(const Bucket& b, char* ws) {
  Bucket32Ptrs q;
  const long long cnt = static_cast<long long>(b.members.size());
  q.xs = cnt * b.m_pad * b.n_pad;
  q.as = cnt * b.m_pad * b.m_pad;
  q.x[0] = reinterpret_cast<float*>(ws + b.off_x0);
  q.x[1] = reinterpret_cast<float*>(ws + b.off_x1);
  q.a = reinterpret_cast<float*>(ws + b.off_a);
  q.b = reinterpret_cast<float*>(ws + b.off_b);
  return q;
}

// 3-D fp32 tensor map over [count][outer][inner], box {32, 128, 1}, 128-byte swizzle.
int make_map32(CUtensorMap* m, void* base, uint64_t inner, uint64_t outer, uint64_t count) {
  cuuint64_t dims[3] = {inner, outer, count};
  cuuint64_t strides[2] = {inner * 4, inner * outer * 4};
  cuuint32_t box[3] = {32, 128, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? NS_OK : NS_ERR_CUDA;
}

template <typename P>
int fill_phase32(P& gp, const Plan& p, char* ws, int phase, int cur, size_t b0, size_t b1, unsigned int* status,
                 void* const* final_out) {
  std::memset(&gp, 0, sizeof(gp));
  gp.alpha = p.a;
  gp.beta = p.b;
  gp.gamma = p.c;
  gp.status = status;
  long long tiles = 0;
  int nb = 0, n_out = 0;
  for (size_t bi = b0; bi < b1; ++bi, ++nb) {
    const Bucket& b = p.buckets[bi];
    const Bucket32Ptrs q = bucket32_ptrs(b, ws);
    const uint64_t cnt = b.members.size();
    nsk::Gemm32Bucket& g = gp.bk[nb];
    g.tile_begin = tiles;
    g.count = static_cast<int>(cnt);
    g.m_valid = static_cast<int>(b.m);
    g.n_valid = static_cast<int>(b.n);
    g.cols_valid = static_cast<int>(b.m_pad);
    int rc = NS_OK;
    if (phase == nsk::PH32_GRAM || phase == nsk::PH32_A2B) {
      g.tiles_m = static_cast<int>(b.m_pad / nsk::GEMM_BM);
      g.tiles_n = static_cast<int>((b.m_pad + nsk::GEMM_BN - 1) / nsk::GEMM_BN);
      g.tiles_per_mat = static_cast<int>(syrk_tiles(g.tiles_m, g.tiles_n));
      g.ld = static_cast<int>(b.m_pad);
      g.mat_stride = b.m_pad * b.m_pad;
      if (phase == nsk::PH32_GRAM) {
        float* xh = q.x[cur];
        float* xl = xh + q.xs;
        g.k_blocks = static_cast<int>(b.n_pad / 32);
        g.out_h = q.a;
        g.out_l = q.a + q.as;
        rc = make_map32(&gp.tmah[nb], xh, b.n_pad, b.m_pad, cnt);
        if (rc == NS_OK) rc = make_map32(&gp.tmal[nb], xl, b.n_pad, b.m_pad, cnt);
        if (rc == NS_OK) rc = make_map32(&gp.tmbh[nb], xh, b.n_pad, b.m_pad, cnt);
        if (rc == NS_OK) rc = make_map32(&gp.tmbl[nb], xl, b.n_pad, b.m_pad, cnt);
      } else {
        g.k_blocks = static_cast<int>(b.m_pad / 32);
        g.out_h = q.b;
        g.out_l = q.b + q.as;
        g.aux_h = q.a;
        g.aux_l = q.a + q.as;
        g.delta = 0.0f;
        g.beta = p.b;
        g.gamma = p.c;
        rc = make_map32(&gp.tmah[nb], q.a, b.m_pad, b.m_pad, cnt);
        if (rc == NS_OK) rc = make_map32(&gp.tmal[nb], q.a + q.as, b.m_pad, b.m_pad, cnt);
        if (rc == NS_OK) rc = make_map32(&gp.tmbh[nb], q.a, b.m_pad, b.m_pad, cnt);
        if (rc == NS_OK) rc = make_map32(&gp.tmbl[nb], q.a + q.as, b.m_pad, b.m_pad, cnt);
      }
    } else {
      // (B X)^T = X^T B: M over n (X^T rows), N over m (B rows), K = m
      float* xc = q.x[cur];
      float* xn = q.x[1 - cur];
      g.tiles_m = static_cast<int>(b.n_pad / nsk::GEMM_BM);
      g.tiles_n = static_cast<int>((b.m_pad + nsk::GEMM_BN - 1) / nsk::GEMM_BN);
      g.tiles_per_mat = g.tiles_m * g.tiles_n;
      g.k_blocks = static_cast<int>(b.m_pad / 32);
      g.ld = static_cast<int>(b.n_pad);
      g.ld_t = static_cast<int>(b.m_pad);
      g.mat_stride = b.m_pad * b.n_pad;
      g.mat_stride_t = b.m_pad * b.n_pad;
      g.aux_h = xc;
      g.aux_l = xc + q.xs;
      g.out_h = xn;
      g.out_l = xn + q.xs;
      g.out_th = xn + 2 * q.xs;
      g.out_tl = xn + 3 * q.xs;
      rc = make_map32(&gp.tmah[nb], xc + 2 * q.xs, b.m_pad, b.n_pad, cnt);
      if (rc == NS_OK) rc = make_map32(&gp.tmal[nb], xc + 3 * q.xs, b.m_pad, b.n_pad, cnt);
      if (rc == NS_OK) rc = make_map32(&gp.tmbh[nb], q.b, b.m_pad, b.m_pad, cnt);
      if (rc == NS_OK) rc = make_map32(&gp.tmbl[nb], q.b + q.as, b.m_pad, b.m_pad, cnt);
      if (final_out) {
        g.out_first = n_out;
        for (size_t s = 0; s < cnt; ++s) {
          const Tensor& t = p.t[b.members[s]];
          const unsigned long long a = reinterpret_cast<unsigned long long>(final_out[t.ordinal]);
          gp.out_tab[n_out++] = a | (t.transposed ? 1ull : 0ull);
        }
      }
    }
    if (rc != NS_OK) return rc;
    tiles += static_cast<long long>(g.tiles_per_mat) * static_cast<long long>(cnt);
  }
  gp.nb = nb;
  gp.total_tiles = tiles;
  return NS_OK;
}

// ------------------------------------------------- fp32 Gram-space path
// Per bucket: the X_0 set in the first X region; A and Q in the A and B
// regions; T, P0, P1 (hi, lo pairs of m_pad^2) in the second X region.
struct GsPtrs {
  float* a;
  float* q;
  float* t;
  float* p[2];
  float* coef;
  long long as;
};

GsPtrs gs_ptrs(const Bucket& b, char* ws) {
  const Bucket32Ptrs q = bucket32_ptrs(b, ws);
  GsPtrs g;
  g.as = q.as;
  g.a = q.a;
  g.q = q.b;
  float* x1 = reinterpret_cast<float*>(ws + b.off_x1);
  g.t = x1;
  g.p[0] = x1 + 2 * q.as;
  g.p[1] = x1 + 4 * q.as;
  g.coef = reinterpret_cast<float*>(ws + b.off_coef);
  return g;
}

// One launch of D = delta*I + beta*Aux + gamma*(L R) (L, R symmetric and
// commuting, so D is symmetric: upper tiles + mirror) over buckets [b0, b1).
// sel(bucket, which) returns the hi pointer of operand `which` (0 = L, 1 = R,
// 2 = Aux or null, 3 = output); coefs per matrix when `per_matrix`.
template <typename Sel>
int run_sym32(const Plan& p, char* ws, size_t b0, size_t b1, Sel sel, float delta, float beta, float gamma,
              bool per_matrix, int nsm, unsigned int* status, cudaStream_t st) {
  nsk::Gemm32Params gp;
  std::memset(&gp, 0, sizeof(gp));
  gp.status = status;
  long long tiles = 0;
  int nb = 0;
  for (size_t bi = b0; bi < b1; ++bi, ++nb) {
    const Bucket& b = p.buckets[bi];
    const GsPtrs gs = gs_ptrs(b, ws);
    const uint64_t cnt = b.members.size();
    nsk::Gemm32Bucket& g = gp.bk[nb];
    g.tile_begin = tiles;
    g.count = static_cast<int>(cnt);
    g.m_valid = static_cast<int>(b.m);
    g.n_valid = static_cast<int>(b.n);
    g.cols_valid = static_cast<int>(b.m_pad);
    g.tiles_m = static_cast<int>(b.m_pad / nsk::GEMM_BM);
    g.tiles_n = static_cast<int>((b.m_pad + nsk::GEMM_BN - 1) / nsk::GEMM_BN);
    g.tiles_per_mat = static_cast<int>(syrk_tiles(g.tiles_m, g.tiles_n));
    g.ld = static_cast<int>(b.m_pad);
    g.mat_stride = b.m_pad * b.m_pad;
    g.k_blocks = static_cast<int>(b.m_pad / 32);
    float* L = sel(bi, 0);
    float* R = sel(bi, 1);
    float* X = sel(bi, 2);
    float* O = sel(bi, 3);
    g.out_h = O;
    g.out_l = O + gs.as;
    g.aux_h = X;
    g.aux_l = X ? X + gs.as : nullptr;
    g.coef = per_matrix ? gs.coef : nullptr;
    g.delta = delta;
    g.beta = beta;
    g.gamma = gamma;
    int rc = make_map32(&gp.tmah[nb], L, b.m_pad, b.m_pad, cnt);
    if (rc == NS_OK) rc = make_map32(&gp.tmal[nb], L + gs.as, b.m_pad, b.m_pad, cnt);
    if (rc == NS_OK) rc = make_map32(&gp.tmbh[nb], R, b.m_pad, b.m_pad, cnt);
    if (rc == NS_OK) rc = make_map32(&gp.tmbl[nb], R + gs.as, b.m_pad, b.m_pad, cnt);
    if (rc != NS_OK) return rc;
    tiles += static_cast<long long>(g.tiles_per_mat) * static_cast<long long>(cnt);
  }
  gp.nb = nb;
  gp.total_tiles = tiles;
  const int grid = static_cast<int>(std::min<long long>(gp.total_tiles, nsm));
  return counted(nsk::PH32_A2B, st, [&] { return nsk::launch_gemm32(nsk::PH32_A2B, gp, grid, st); }) ==
                 cudaSuccess
             ? NS_OK
             : NS_ERR_CUDA;
}

int orthogonalize_f32(const Plan& p, const void* const* in, void* const* out, char* ws, int nsm,
                      unsigned int* status, cudaStream_t st);

int orthogonalize_gram_space(const Plan& p, const void* const* in, void* const* out, char* ws, int nsm,
                             unsigned int* status, cudaStream_t st) {
  // prologue and A_0 = X_0 X_0^T as in the fp32 path: run the fp32 prologue
  // through its first Gram by asking it for zero further steps is not
  // possible, so the pieces are launched here directly.
  for (const Bucket& b : p.buckets) {
    const BucketPtrs q0 = bucket_ptrs(b, ws);
    const Bucket32Ptrs q = bucket32_ptrs(b, ws);
    const size_t cnt = b.members.size();
    for (size_t s0 = 0; s0 < cnt; s0 += nsk::PRO_MAX_MATS) {
      nsk::ProParams pp;
      std::memset(&pp, 0, sizeof(pp));
      pp.count = static_cast<int>(std::min<size_t>(nsk::PRO_MAX_MATS, cnt - s0));
      pp.nchunks = static_cast<int>(b.nchunks);
      pp.m_pad = static_cast<int>(b.m_pad);
      pp.n_pad = static_cast<int>(b.n_pad);
      pp.m = static_cast<int>(b.m);
      pp.n = static_cast<int>(b.n);
      pp.eps = p.eps;
      pp.out_f32 = 1;
      pp.x_split = q.xs;
      pp.status = status;
      for (int k = 0; k < pp.count; ++k) {
        const size_t s = s0 + k;
        const Tensor& t = p.t[b.members[s]];
        nsk::MatDesc& d = pp.md[k];
        d.in = in[t.ordinal];
        d.out = out[t.ordinal];
        d.x = q.x[0] + s * b.m_pad * b.n_pad;
        d.partial = q0.partial + s * b.nchunks;
        d.scale = q0.scale + s;
        d.numel = t.numel;
        d.rows = static_cast<int>(t.rows);
        d.cols = static_cast<int>(t.cols);
        d.transposed = t.transposed ? 1 : 0;
      }
      if (counted(K_PRO, st, [&] { return nsk::launch_sumsq(pp, st); }) != cudaSuccess ||
          counted(K_PRO, st, [&] { return nsk::launch_scale(pp, st); }) != cudaSuccess ||
          counted(K_PRO, st, [&] { return nsk::launch_prep32(pp, st); }) != cudaSuccess)
        return NS_ERR_CUDA;
    }
  }
  std::vector<int> pcur(p.buckets.size(), 0);
  for (size_t b0 = 0; b0 < p.buckets.size(); b0 += nsk::GEMM_MAX_BUCKETS) {
    const size_t b1 = std::min(p.buckets.size(), b0 + nsk::GEMM_MAX_BUCKETS);
    // A_0 = X_0 X_0^T
    {
      nsk::Gemm32Params gp;
      int rc = fill_phase32(gp, p, ws, nsk::PH32_GRAM, 0, b0, b1, status, nullptr);
      if (rc != NS_OK) return rc;
      const int grid = static_cast<int>(std::min<long long>(gp.total_tiles, nsm));
      if (counted(nsk::PH32_GRAM, st, [&] { return nsk::launch_gemm32(nsk::PH32_GRAM, gp, grid, st); }) !=
          cudaSuccess)
        return NS_ERR_CUDA;
    }
    const bool ridge = p.ridge > 0.0f;
    for (int step = 0; step < p.steps; ++step) {
      if (ridge) {
        // per-matrix Q coefficients from r = ridge * tr(A) / m
        nsk::Ridge32Params rp;
        std::memset(&rp, 0, sizeof(rp));
        rp.ridge = p.ridge;
        rp.a = p.a;
        rp.b = p.b;
        rp.c = p.c;
        for (size_t bi = b0; bi < b1; ++bi) {
          const Bucket& b = p.buckets[bi];
          const GsPtrs gs = gs_ptrs(b, ws);
          nsk::Ridge32Bucket& r = rp.bk[rp.nb];
          r.ah = gs.a;
          r.al = gs.a + gs.as;
          r.mat_stride = b.m_pad * b.m_pad;
          r.ld = static_cast<int>(b.m_pad);
          r.m = static_cast<int>(b.m);
          r.count = static_cast<int>(b.members.size());
          rp.coef[rp.nb] = gs.coef;
          rp.max_count = std::max(rp.max_count, r.count);
          ++rp.nb;
        }
        if (counted(K_PRO, st, [&] { return nsk::launch_ridge32(rp, st); }) != cudaSuccess) return NS_ERR_CUDA;
      }
      // Q = delta I + beta A + gamma A A
      int rc = run_sym32(
          p, ws, b0, b1,
          [&](size_t bi, int w) -> float* {
            const GsPtrs gs = gs_ptrs(p.buckets[bi], ws);
            return w == 3 ? gs.q : gs.a;
          },
          p.a, p.b, p.c, ridge, nsm, status, st);
      if (rc != NS_OK) return rc;
      if (step == 0) {
        // P_1 = Q_0
        for (size_t bi = b0; bi < b1; ++bi) {
          const GsPtrs gs = gs_ptrs(p.buckets[bi], ws);
          if (cudaMemcpyAsync(gs.p[pcur[bi]], gs.q, 2 * gs.as * sizeof(float), cudaMemcpyDeviceToDevice, st) !=
              cudaSuccess)
            return NS_ERR_CUDA;
        }
      } else {
        // P <- Q P
        rc = run_sym32(
            p, ws, b0, b1,
            [&](size_t bi, int w) -> float* {
              const GsPtrs gs = gs_ptrs(p.buckets[bi], ws);
              return w == 0 ? gs.q : w == 1 ? gs.p[pcur[bi]] : w == 2 ? nullptr : gs.p[1 - pcur[bi]];
            },
            0.0f, 0.0f, 1.0f, false, nsm, status, st);
        if (rc != NS_OK) return rc;
        for (size_t bi = b0; bi < b1; ++bi) pcur[bi] = 1 - pcur[bi];
      }
      if (step + 1 < p.steps) {
        // T = Q A, then A <- Q T (= Q A Q)
        rc = run_sym32(
            p, ws, b0, b1,
            [&](size_t bi, int w) -> float* {
              const GsPtrs gs = gs_ptrs(p.buckets[bi], ws);
              return w == 0 ? gs.q : w == 1 ? gs.a : w == 2 ? nullptr : gs.t;
            },
            0.0f, 0.0f, 1.0f, false, nsm, status, st);
        if (rc != NS_OK) return rc;
        rc = run_sym32(
            p, ws, b0, b1,
            [&](size_t bi, int w) -> float* {
              const GsPtrs gs = gs_ptrs(p.buckets[bi], ws);
              return w == 0 ? gs.q : w == 1 ? gs.t : w == 2 ? nullptr : gs.a;
            },
            0.0f, 0.0f, 1.0f, false, nsm, status, st);
        if (rc != NS_OK) return rc;
      }
    }
    // X_k = P X_0, stored straight to the outputs when the table fits
    if (p.steps == 0) continue;
    if (group_matrices(p, b0, b1) <= size_t(nsk::GEMM32_MAX_OUT)) {
      static thread_local nsk::Gemm32FinalParams gp;
      int rc = fill_phase32(gp, p, ws, nsk::PH32_BXT, 0, b0, b1, status, out);
      if (rc != NS_OK) return rc;
      gp.alpha = 0.0f;
      int nb = 0;
      for (size_t bi = b0; bi < b1; ++bi, ++nb) {
        const Bucket& b = p.buckets[bi];
        const GsPtrs gs = gs_ptrs(b, ws);
        const uint64_t cnt = b.members.size();
        rc = make_map32(&gp.tmbh[nb], gs.p[pcur[bi]], b.m_pad, b.m_pad, cnt);
        if (rc == NS_OK) rc = make_map32(&gp.tmbl[nb], gs.p[pcur[bi]] + gs.as, b.m_pad, b.m_pad, cnt);
        if (rc != NS_OK) return rc;
      }
      const int grid = static_cast<int>(std::min<long long>(gp.total_tiles, nsm));
      if (counted(K_BX_FINAL, st, [&] { return nsk::launch_gemm32_final(gp, grid, st); }) != cudaSuccess)
        return NS_ERR_CUDA;
    } else {
      return NS_ERR_UNSUPPORTED;  // more matrices than one final launch can address
    }
  }
  if (p.steps == 0) {
    // X_0 itself: reuse the fp32 path, which stores X_0 when steps == 0
    return orthogonalize_f32(p, in, out, ws, nsm, status, st);
  }
  return NS_OK;
}

int orthogonalize_f32(const Plan& p, const void* const* in, void* const* out, char* ws, int nsm,
                      unsigned int* status, cudaStream_t st) {
  // prologue: sums of squares, scales, X_0 hi/lo in both orientations
  for (const Bucket& b : p.buckets) {
    const BucketPtrs q0 = bucket_ptrs(b, ws);
    const Bucket32Ptrs q = bucket32_ptrs(b, ws);
    const size_t cnt = b.members.size();
    for (size_t s0 = 0; s0 < cnt; s0 += nsk::PRO_MAX_MATS) {
      nsk::ProParams pp;
      std::memset(&pp, 0, sizeof(pp));
      pp.count = static_cast<int>(std::min<size_t>(nsk::PRO_MAX_MATS, cnt - s0));
      pp.nchunks = static_cast<int>(b.nchunks);
      pp.m_pad = static_cast<int>(b.m_pad);
      pp.n_pad = static_cast<int>(b.n_pad);
      pp.m = static_cast<int>(b.m);
      pp.n = static_cast<int>(b.n);
      pp.eps = p.eps;
      pp.out_f32 = 1;
      pp.x_split = q.xs;
      pp.status = status;
      for (int k = 0; k < pp.count; ++k) {
        const size_t s = s0 + k;
        const Tensor& t = p.t[b.members[s]];
        nsk::MatDesc& d = pp.md[k];
        d.in = in[t.ordinal];
        d.out = out[t.ordinal];
        d.x = q.x[0] + s * b.m_pad * b.n_pad;
        d.partial = q0.partial + s * b.nchunks;
        d.scale = q0.scale + s;
        d.numel = t.numel;
        d.rows = static_cast<int>(t.rows);
        d.cols = static_cast<int>(t.cols);
        d.transposed = t.transposed ? 1 : 0;
      }
      if (counted(K_PRO, st, [&] { return nsk::launch_sumsq(pp, st); }) != cudaSuccess ||
          counted(K_PRO, st, [&] { return nsk::launch_scale(pp, st); }) != cudaSuccess ||
          counted(K_PRO, st, [&] { return nsk::launch_prep32(pp, st); }) != cudaSuccess)
        return NS_ERR_CUDA;
    }
  }
  std::vector<char> stored(p.buckets.size(), 0);
  int cur = 0;
  for (int step = 0; step < p.steps; ++step) {
    const bool last = step + 1 == p.steps;
    for (int phase = nsk::PH32_GRAM; phase <= nsk::PH32_BXT; ++phase) {
      for (size_t b0 = 0; b0 < p.buckets.size(); b0 += nsk::GEMM_MAX_BUCKETS) {
        const size_t b1 = std::min(p.buckets.size(), b0 + nsk::GEMM_MAX_BUCKETS);
        int rc;
        if (last && phase == nsk::PH32_BXT && group_matrices(p, b0, b1) <= size_t(nsk::GEMM32_MAX_OUT)) {
          static thread_local nsk::Gemm32FinalParams gp;
          rc = fill_phase32(gp, p, ws, phase, cur, b0, b1, status, out);
          if (rc != NS_OK) return rc;
          const int grid = static_cast<int>(std::min<long long>(gp.total_tiles, nsm));
          if (counted(K_BX_FINAL, st, [&] { return nsk::launch_gemm32_final(gp, grid, st); }) != cudaSuccess)
            return NS_ERR_CUDA;
          for (size_t bi = b0; bi < b1; ++bi) stored[bi] = 1;
        } else {
          nsk::Gemm32Params gp;
          rc = fill_phase32(gp, p, ws, phase, cur, b0, b1, status, nullptr);
          if (rc != NS_OK) return rc;
          const int grid = static_cast<int>(std::min<long long>(gp.total_tiles, nsm));
          if (counted(phase, st, [&] { return nsk::launch_gemm32(phase, gp, grid, st); }) != cudaSuccess)
            return NS_ERR_CUDA;
        }
        if (phase == nsk::PH32_GRAM && p.ridge > 0.0f) {
          nsk::Ridge32Params rp;
          std::memset(&rp, 0, sizeof(rp));
          rp.ridge = p.ridge;
          for (size_t bi = b0; bi < b1; ++bi) {
            const Bucket& b = p.buckets[bi];
            const Bucket32Ptrs q = bucket32_ptrs(b, ws);
            nsk::Ridge32Bucket& r = rp.bk[rp.nb++];
            r.ah = q.a;
            r.al = q.a + q.as;
            r.mat_stride = b.m_pad * b.m_pad;
            r.ld = static_cast<int>(b.m_pad);
            r.m = static_cast<int>(b.m);
            r.count = static_cast<int>(b.members.size());
            rp.max_count = std::max(rp.max_count, r.count);
          }
          if (counted(K_PRO, st, [&] { return nsk::launch_ridge32(rp, st); }) != cudaSuccess) return NS_ERR_CUDA;
        }
      }
    }
    cur = 1 - cur;
  }
  for (size_t bi = 0; bi < p.buckets.size(); ++bi) {
    if (stored[bi]) continue;
    const Bucket& b = p.buckets[bi];
    const Bucket32Ptrs q = bucket32_ptrs(b, ws);
    const size_t cnt = b.members.size();
    for (size_t s0 = 0; s0 < cnt; s0 += nsk::PRO_MAX_MATS) {
      nsk::ProParams pp;
      std::memset(&pp, 0, sizeof(pp));
      pp.count = static_cast<int>(std::min<size_t>(nsk::PRO_MAX_MATS, cnt - s0));
      pp.m_pad = static_cast<int>(b.m_pad);
      pp.n_pad = static_cast<int>(b.n_pad);
      pp.m = static_cast<int>(b.m);
      pp.n = static_cast<int>(b.n);
      pp.out_f32 = 1;
      pp.x_split = q.xs;
      pp.status = status;
      for (int k = 0; k < pp.count; ++k) {
        const size_t s = s0 + k;
        const Tensor& t = p.t[b.members[s]];
        nsk::MatDesc& d = pp.md[k];
        d.out = out[t.ordinal];
        d.xfinal = q.x[cur] + s * b.m_pad * b.n_pad;
        d.rows = static_cast<int>(t.rows);
        d.cols = static_cast<int>(t.cols);
        d.transposed = t.transposed ? 1 : 0;
        d.numel = t.numel;
      }
      if (counted(K_PRO, st, [&] { return nsk::launch_store32(pp, st); }) != cudaSuccess) return NS_ERR_CUDA;
    }
  }
  return NS_OK;
}

// bf16 path, part 1: sums of squares, scales, X_0 = scale * (T or T^T),
// zero padded into the workspace.
// With rank_in (row-shard plans, shard_dim 0) the rows are read straight from
// the S rank buffers, which fuses the pack to the home buffers away; `in` is
// then unused.
int prologue_bf16(const Plan& p, const void* const* in, void* const* out, char* ws, unsigned int* status,
                  cudaStream_t st, const void* const* rank_in = nullptr) {
  // prologue: X~_0 = T or T^T (unscaled, zero padded) with per-stripe sums of
  // squares in one pass, then the scales
  for (const Bucket& b : p.buckets) {
    const BucketPtrs q = bucket_ptrs(b, ws);
    const size_t cnt = b.members.size();
    for (size_t s0 = 0; s0 < cnt; s0 += nsk::PRO_MAX_MATS) {
      nsk::ProParams pp;
      std::memset(&pp, 0, sizeof(pp));
      pp.count = static_cast<int>(std::min<size_t>(nsk::PRO_MAX_MATS, cnt - s0));
      pp.nchunks = static_cast<int>(b.nchunks);
      pp.m_pad = static_cast<int>(b.m_pad);
      pp.n_pad = static_cast<int>(b.n_pad);
      pp.m = static_cast<int>(b.m);
      pp.n = static_cast<int>(b.n);
      pp.eps = p.eps;
      pp.out_f32 = 0;
      pp.status = status;
      if (rank_in) {
        pp.from_ranks = 1;
        pp.ranks_aligned = 1;
        for (int r = 0; r < p.S; ++r) {
          pp.rank_ptr[r] = rank_in[r];
          if (reinterpret_cast<uintptr_t>(rank_in[r]) & 15) pp.ranks_aligned = 0;
        }
      }
      for (int k = 0; k < pp.count; ++k) {
        const size_t s = s0 + k;
        const Tensor& t = p.t[b.members[s]];
        nsk::MatDesc& d = pp.md[k];
        d.in = rank_in ? nullptr : in[t.ordinal];
        d.rank_off = t.rank_off;
        d.shard_rows = static_cast<int>(t.rows / p.S);
        d.out = out[t.ordinal];
        d.x = q.x0 + s * b.m_pad * b.n_pad * 2;
        d.partial = q.partial + s * b.nchunks;
        d.scale = q.scale + s;
        d.numel = t.numel;
        d.rows = static_cast<int>(t.rows);
        d.cols = static_cast<int>(t.cols);
        d.transposed = t.transposed ? 1 : 0;
      }
      if (counted(K_PRO, st, [&] { return nsk::launch_prep(pp, st); }) != cudaSuccess ||
          counted(K_PRO, st, [&] { return nsk::launch_scale(pp, st); }) != cudaSuccess)
        return NS_ERR_CUDA;
    }
  }
  return NS_OK;
}

// Whether every bucket group's last B*X launch can store its results itself
// (its per-matrix table fits the parameter block) and there is a last step.
bool final_stores_all(const Plan& p) {
  if (p.steps == 0) return false;
  for (size_t b0 = 0; b0 < p.buckets.size(); b0 += nsk::GEMM_MAX_BUCKETS)
    if (group_matrices(p, b0, std::min(p.buckets.size(), b0 + nsk::GEMM_MAX_BUCKETS)) > size_t(nsk::GEMM_MAX_OUT))
      return false;
  return true;
}

// bf16 path, part 2: k steps of (Gram, A*A + B, B*X) and the final store.
// With rank_out (row shards along dim 0, final_stores_all(p)) the results go
// straight to the S rank buffers, fusing the unpack away; `out` is then unused.
int steps_bf16(const Plan& p, void* const* out, char* ws, int nsm, unsigned int* status, cudaStream_t st,
               void* const* rank_out = nullptr) {
  if (rank_out && !final_stores_all(p)) return NS_ERR_ARG;
  int rc = NS_OK;
  // k steps x (Gram, A*A + B, B*X) over all buckets. The last B*X launch of
  // a bucket group writes the results straight to `out` when its per-matrix
  // table fits the parameter block; other groups go through the store kernel.
  std::vector<char> stored(p.buckets.size(), 0);
  bool cur_is_x0 = true;
  for (int step = 0; step < p.steps; ++step) {
    const bool last = step + 1 == p.steps;
    for (int phase = nsk::PH_GRAM; phase <= nsk::PH_BX; ++phase) {
      for (size_t b0 = 0; b0 < p.buckets.size(); b0 += nsk::GEMM_MAX_BUCKETS) {
        const size_t b1 = std::min(p.buckets.size(), b0 + nsk::GEMM_MAX_BUCKETS);
        // serpentine order: every other product walks its tiles backwards,
        // starting on the matrices the previous product wrote last (still in L2)
        const bool serp = ((step * 3 + phase) & 1) != 0;
        if (last && phase == nsk::PH_BX && group_matrices(p, b0, b1) <= size_t(nsk::GEMM_MAX_OUT)) {
          rc = run_final_bx(p, ws, cur_is_x0, b0, b1, nsm, status, out, step == 0, serp, st, rank_out);
          for (size_t bi = b0; bi < b1; ++bi) stored[bi] = 1;
        } else {
          rc = run_phase(p, ws, phase, cur_is_x0, b0, b1, nsm, status, step == 0, serp, st);
        }
        if (rc != NS_OK) return rc;
      }
    }
    cur_is_x0 = !cur_is_x0;
  }
  // transpose back and store (buckets not stored by the last B*X launch)
  for (size_t bi = 0; bi < p.buckets.size(); ++bi) {
    if (stored[bi]) continue;
    const Bucket& b = p.buckets[bi];
    const BucketPtrs q = bucket_ptrs(b, ws);
    const char* xf = cur_is_x0 ? q.x0 : q.x1;
    const size_t cnt = b.members.size();
    for (size_t s0 = 0; s0 < cnt; s0 += nsk::PRO_MAX_MATS) {
      nsk::ProParams pp;
      std::memset(&pp, 0, sizeof(pp));
      pp.count = static_cast<int>(std::min<size_t>(nsk::PRO_MAX_MATS, cnt - s0));
      pp.m_pad = static_cast<int>(b.m_pad);
      pp.n_pad = static_cast<int>(b.n_pad);
      pp.m = static_cast<int>(b.m);
      pp.n = static_cast<int>(b.n);
      pp.out_f32 = p.out_bytes == 4 ? 1 : 0;
      pp.apply_scale = p.steps == 0 ? 1 : 0;  // X~_0 itself, still unscaled
      pp.status = status;
      for (int k = 0; k < pp.count; ++k) {
        const size_t s = s0 + k;
        const Tensor& t = p.t[b.members[s]];
        nsk::MatDesc& d = pp.md[k];
        d.out = out[t.ordinal];
        d.scale = q.scale + s;
        d.xfinal = xf + s * b.m_pad * b.n_pad * 2;
        d.rows = static_cast<int>(t.rows);
        d.cols = static_cast<int>(t.cols);
        d.transposed = t.transposed ? 1 : 0;
        d.numel = t.numel;
      }
      if (counted(K_PRO, st, [&] { return nsk::launch_store(pp, st); }) != cudaSuccess) return NS_ERR_CUDA;
    }
  }
  return NS_OK;
}

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

int pipe_device(ns_pipeline* pl, int d) {
  PipeDev& pd = pl->dev[d];
  if (pd.mem) return NS_OK;
  if (cudaStreamCreateWithFlags(&pd.mem, cudaStreamNonBlocking) != cudaSuccess ||
      cudaStreamCreateWithFlags(&pd.gemm, cudaStreamNonBlocking) != cudaSuccess ||
      cudaStreamCreateWithFlags(&pd.out, cudaStreamNonBlocking) != cudaSuccess)
    return NS_ERR_CUDA;
  pd.ev.assign(4 + 2 * pl->W, nullptr);
  for (cudaEvent_t& e : pd.ev)
    if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return NS_ERR_CUDA;
  return NS_OK;
}

}  // namespace

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
  return steps_bf16(p, out, ws, nsm, status, st);
}

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
  if (cl < 0 || cl > 3) return NS_ERR_ARG;
  std::lock_guard<std::mutex> lk(g_mu);
  g_force_cl = cl;
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


int ns_pipeline_create(ns_plan_t* plan, int n_waves, ns_pipeline_t** out) {
  if (!out) return NS_ERR_ARG;
  *out = nullptr;
  if (!plan || n_waves < 1) return NS_ERR_ARG;
  const Plan& p = plan->p;
  if (p.gram_mode != NS_BF16) return NS_ERR_UNSUPPORTED;
  const int np = static_cast<int>(p.part.size());
  const int W = std::max(1, std::min(n_waves, np));
  ns_pipeline* pl = new (std::nothrow) ns_pipeline();
  if (!pl) return NS_ERR_ARG;
  pl->base = plan;
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
      for (cudaEvent_t e : pd.ev)
        if (e) cudaEventDestroy(e);
      cudaStreamDestroy(pd.mem);
      cudaStreamDestroy(pd.gemm);
      cudaStreamDestroy(pd.out);
    }
    if (have) cudaSetDevice(cur);
  }
  delete pl;
  return NS_OK;
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
