// Host orchestration shared by the device-side C ABI files (api.cu,
// runtime.cu, route.cu, ns_bf16.cu, ns_fp32.cu, pipeline.cu): per-device set-up
// and status word, launch counting and timing, tensor maps, the bf16 and fp32
// Newton-Schulz orchestration and the routing between rank and home buffers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "../../include/nsgb300.h"
#include "kernels.h"
#include "plan.h"

namespace nsorch {

using nsplan::Bucket;
using nsplan::Plan;
using nsplan::Tensor;

// ------------------------------------------------------------ runtime.cu
// Per-device set-up: status word address, SM count, architecture check.
int device_setup(int* dev_out, unsigned int** status_out, int* nsm_out);
// GEMM tiling forced by ns_set_gemm_cluster (0: automatic).
int gemm_cluster_override();
// Whether buckets marked small run as one CTA per matrix (ns_set_small_path).
bool small_path_enabled();
// Whether the bf16 symmetric products store their mirror (ns_set_symmetric_store).
bool symmetric_mirror();
// Test support: the wait limit armed by ns_test_stall_next_gemm (0 if none),
// cleared by this call; the launch that takes it stalls.
unsigned long long take_gemm_stall();

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
// cuTensorMapEncodeTiled, looked up by device_setup.
EncodeTiledFn tensor_map_encoder();

// 3-D bf16 tensor map over [count][outer][inner] with a {box_inner, box_outer, 1}
// box, 128-byte swizzle (operand tiles) or 64-byte swizzle (epilogue chunks of
// 32 x 32), zero fill outside the array.
int make_map(CUtensorMap* m, void* base, uint64_t inner, uint64_t outer, uint64_t count, uint32_t box_inner,
             uint32_t box_outer, CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B);
int make_epi_map(CUtensorMap* m, void* base, uint64_t inner, uint64_t outer, uint64_t count);

// Launch kinds of ns_profile_read.
constexpr int kKinds = 7;
enum { K_GRAM = 0, K_A2B = 1, K_BX = 2, K_PRO = 3, K_PACK = 4, K_BX_FINAL = 5, K_SMALL = 6 };
// Count a launch of `kind`; when timing is on, hand out two events for it.
bool prof_begin(int kind, cudaEvent_t* a, cudaEvent_t* b);
// Queue the bracketing events of a timed launch for ns_profile_read.
void prof_end(int kind, cudaEvent_t a, cudaEvent_t b);

// Launch through `fn`, counting it and, if timing is on, bracketing it with
// events on `st`.
template <typename F>
cudaError_t counted(int kind, cudaStream_t st, F&& fn) {
  cudaEvent_t a = nullptr, b = nullptr;
  const bool timed = prof_begin(kind, &a, &b);
  if (timed && a) cudaEventRecord(a, st);
  cudaError_t e = fn();
  if (timed && b) {
    cudaEventRecord(b, st);
    prof_end(kind, a, b);
  }
  return e;
}

// ------------------------------------------------------------ ns_bf16.cu
struct BucketPtrs {
  char* x0;
  char* x1;
  char* a;
  char* b;
  float* partial;
  float* scale;
};
BucketPtrs bucket_ptrs(const Bucket& b, char* ws);
// Upper-triangle work items of one matrix (cl = 1: single tiles; else pairs).
long long syrk_tiles(int tiles_m, int tiles_n, int cl = 1);
// Matrices of the bucket group [b0, b1).
size_t group_matrices(const Plan& p, size_t b0, size_t b1);
// bf16 prologue: X~_0 (unscaled, padded, transposed where needed) and the
// scales; with rank_in (row shards along dim 0) the rows come straight from
// the S rank buffers.
int prologue_bf16(const Plan& p, const void* const* in, void* const* out, char* ws, unsigned int* status,
                  cudaStream_t st, const void* const* rank_in = nullptr);
// Buckets [0, gemm_buckets(p)) run through the GEMM launches; the rest (small
// buckets, when the one-CTA-per-matrix path is on) through small_bf16.
size_t gemm_buckets(const Plan& p);
// The whole iteration of every small bucket, one CTA per matrix, inputs from
// `in` (or with rank_in from the S rank buffers, row shards along dim 0) and
// results to `out` (or with rank_out to the rank buffers).
int small_bf16(const Plan& p, const void* const* in, void* const* out, unsigned int* status, cudaStream_t st,
               const void* const* rank_in = nullptr, void* const* rank_out = nullptr);
// Whether every bucket group's last B*X launch can store its results itself.
bool final_stores_all(const Plan& p);
// k steps of (Gram, A*A + B, B*X) and the final store (into `out`, or with
// rank_out into the S rank buffers).
int steps_bf16(const Plan& p, void* const* out, char* ws, int nsm, unsigned int* status, cudaStream_t st,
               void* const* rank_out = nullptr);

// ------------------------------------------------------------ ns_fp32.cu
int orthogonalize_f32(const Plan& p, const void* const* in, void* const* out, char* ws, int nsm,
                      unsigned int* status, cudaStream_t st);
int orthogonalize_gram_space(const Plan& p, const void* const* in, void* const* out, char* ws, int nsm,
                             unsigned int* status, cudaStream_t st);

// -------------------------------------------------------------- route.cu
// Pack (to_home) or unpack the entry-coordinate range [g_begin, g_end)
// (g_end < 0: everything).
int route(ns_plan_t* plan, void* const* rank_bufs, void* const* home_bufs, int S, int shard_dim, bool to_home,
          int elem_bytes, cudaStream_t st, long long g_begin = 0, long long g_end = -1);

}  // namespace nsorch
