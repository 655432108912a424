// Whole Newton-Schulz iteration of a small matrix in one CTA (Megatron-Core
// API page owner_planning, ns_cost_fn: view as (shape[0], prod(shape[1:])),
// transpose so rows <= cols, normalise, then per step A = X X^T;
// X = a X + (b A + c A A) X; transposed back at the end).
//
// For m <= 128 and n <= 512 everything fits on one SM: X (128 x n_pad bf16,
// up to 128 KB), A and B (128 x 128 bf16, 32 KB each) stay in shared memory
// and the three products accumulate in TMEM, so a whole call is one launch
// (one CTA per matrix) instead of a prologue, 3k GEMM launches and a store.
//
// Shared-memory layout (128-byte swizzle, the layout a TMA box {64, 128}
// would produce): a matrix of 128 rows is stored as chunks of 64 columns,
// each chunk 128 rows x 128 bytes (16 KB), 16-byte unit u of row r at unit
// u ^ (r & 7). One copy of each matrix serves every product it enters:
//   Gram  A = X X^T : both operands X, K-major (K = n)
//   A*A             : both operands A, K-major (A is symmetric)
//   B*X             : A operand B, K-major; B operand X read MN-major (N = n
//                     contiguous, chunks 16 KB apart, K = m rows)
// TMEM: Gram accumulator in columns [0, 128), A*A in [128, 256), B*X in
// [0, n_pad).
//
// 512 threads (16 warps): in every epilogue warp w owns rows [32 (w % 4), +32)
// (the TMEM lanes that warp may read) and every fourth 32-column chunk starting
// at chunk w / 4, so four warps share each SM sub-partition's work. Thread 0
// issues the MMAs (M = 128, K = 16 per instruction) and commits them to an
// mbarrier that every thread waits on (bounded). The normalisation is folded
// into the first step as in the GEMM path: X~_0 holds the input unscaled, the
// first Gram writes s^2 acc and the first B*X s (a X~ + acc), s = 1/(||T||_F + eps).
#include <cuda_bf16.h>

#include <algorithm>
#include <atomic>
#include <cstddef>
#include <cstring>

#include "kernels.h"
#include "launch.cuh"
#include "ptx.cuh"
#include "status.h"

namespace nsk {
namespace {

using namespace nsptx;

constexpr int SM_THREADS = 512;
constexpr int SM_WARPS = SM_THREADS / 32;
constexpr uint32_t CHUNK = 128 * 128;  // bytes of one 64-column chunk of 128 rows

__host__ __device__ constexpr size_t small_smem_bytes(int n_pad) {
  return 1024 + size_t(n_pad / 64) * CHUNK + 4 * CHUNK + 256;
}

// Byte offset of element (row r, column j) in a chunked, swizzled matrix.
__device__ __forceinline__ uint32_t soff(int r, int j) {
  return static_cast<uint32_t>((j >> 6) * CHUNK + r * 128 + ((((j & 63) >> 3) ^ (r & 7)) << 4) + (j & 7) * 2);
}

__device__ __forceinline__ float bf(unsigned short h) { return __uint_as_float(uint32_t(h) << 16); }

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Address of element (r, 0) of row r of the tensor (original orientation).
template <typename P>
__device__ __forceinline__ const unsigned short* in_row(const P& p, const SmallMat& M, int r) {
  if (!p.in_ranks) return reinterpret_cast<const unsigned short*>(M.in) + static_cast<long long>(r) * M.cols;
  const int sh = M.rows / p.S;
  return reinterpret_cast<const unsigned short*>(p.rank_in[r / sh]) + M.rank_off +
         static_cast<long long>(r % sh) * M.cols;
}
template <typename P>
__device__ __forceinline__ unsigned short* out_row(const P& p, const SmallMat& M, int r) {
  if (!p.out_ranks) return reinterpret_cast<unsigned short*>(M.out) + static_cast<long long>(r) * M.cols;
  const int sh = M.rows / p.S;
  return reinterpret_cast<unsigned short*>(p.rank_out[r / sh]) + M.rank_off + static_cast<long long>(r % sh) * M.cols;
}

// 16-byte asynchronous copy global -> shared (both addresses 16-byte aligned).
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// Wait for the MMA group committed to `bar`; false (for every thread) if any
// thread's bounded wait gave up.
__device__ __forceinline__ bool wait_mma(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                         unsigned int* status) {
  const bool got = mbar_wait(bar, parity, abort_flag, status);
  return __syncthreads_and(got ? 1 : 0) != 0;
}

template <typename P>
__global__ void __launch_bounds__(SM_THREADS, 1) ns_small_kernel(const __grid_constant__ P p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int NPL = p.n_pad;  // the launch's largest n_pad: sizes shared memory and TMEM
  uint8_t* sX = smem;
  uint8_t* sA = sX + (NPL / 64) * CHUNK;
  uint8_t* sB = sA + 2 * CHUNK;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sB + 2 * CHUNK);  // [0] MMA groups, [1] drain
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 2);
  float* red = reinterpret_cast<float*>(tmem_slot + 2);  // SM_WARPS warp partial sums
  volatile int* abort_flag = reinterpret_cast<volatile int*>(red + SM_WARPS);

  if (blockDim.x != SM_THREADS || blockIdx.x >= static_cast<unsigned>(p.count)) {
    if (threadIdx.x == 0) atomicOr(p.status, NS_DEV_BAD_LAUNCH);
    return;
  }
  const int t = threadIdx.x, warp = t / 32, lane = t % 32;
  const int lq = warp & 3, cq = warp >> 2;  // TMEM lane quarter, column quarter
  const int row = 32 * lq + lane;           // the row this thread owns in the epilogues
  const uint32_t tmem_cols = NPL > 256 ? 512u : 256u;
  if (t == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, tmem_cols);
    tmem_relinquish();
  }
  // zero the X region: padding rows and columns stay zero, which keeps every
  // product exact on the padded shape
  for (int i = t; i < (NPL / 64) * int(CHUNK / 16); i += SM_THREADS)
    reinterpret_cast<uint4*>(sX)[i] = make_uint4(0, 0, 0, 0);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  griddep_wait();
  griddep_launch_dependents();

  const SmallMat& M = p.mat[blockIdx.x];
  const bool tr = M.transposed != 0;
  const int m = tr ? M.cols : M.rows, n = tr ? M.rows : M.cols;
  const int npad = (n + 63) / 64 * 64;

  // ---- load X~_0 (transposed where rows > cols), all loads in flight at once
  if (!tr) {
    // rows of the input are rows of X: 16-byte asynchronous copies straight
    // into the swizzled layout (unaligned rows element by element)
    for (int r = warp; r < M.rows; r += SM_THREADS / 32) {
      const unsigned short* src = in_row(p, M, r);
      const bool al = (reinterpret_cast<uintptr_t>(src) & 15) == 0;
      for (int c0 = lane * 8; c0 < M.cols; c0 += 32 * 8) {
        if (al && c0 + 8 <= M.cols) {
          cp_async16(sX + soff(r, c0), src + c0);
        } else {
          for (int k = 0; k < 8 && c0 + k < M.cols; ++k)
            *reinterpret_cast<unsigned short*>(sX + soff(r, c0 + k)) = src[c0 + k];
        }
      }
    }
    cp_async_wait_all();
  } else {
    // rows of the input are columns of X (cols <= 128: lanes 0..15 hold a row's
    // 8-element units): LROWS rows per warp in flight, then scattered
    constexpr int LROWS = 8;
    for (int r0 = warp * LROWS; r0 < M.rows; r0 += SM_THREADS / 32 * LROWS) {
      const int c0 = lane * 8;
      uint4 q[LROWS];
#pragma unroll
      for (int j = 0; j < LROWS; ++j) {
        q[j] = make_uint4(0, 0, 0, 0);
        const int r = r0 + j;
        if (r < M.rows && c0 < M.cols) {
          const unsigned short* src = in_row(p, M, r) + c0;
          if (c0 + 8 <= M.cols && (reinterpret_cast<uintptr_t>(src) & 15) == 0) {
            q[j] = __ldg(reinterpret_cast<const uint4*>(src));
          } else {
            unsigned short* h = reinterpret_cast<unsigned short*>(&q[j]);
            for (int k = 0; k < 8 && c0 + k < M.cols; ++k) h[k] = src[k];
          }
        }
      }
#pragma unroll
      for (int j = 0; j < LROWS; ++j) {
        const int r = r0 + j;
        if (r >= M.rows || c0 >= M.cols) continue;
        const unsigned short* h = reinterpret_cast<const unsigned short*>(&q[j]);
#pragma unroll
        for (int k = 0; k < 8; ++k)
          if (c0 + k < M.cols) *reinterpret_cast<unsigned short*>(sX + soff(c0 + k, r)) = h[k];
      }
    }
  }
  fence_proxy_async_smem();  // X~_0 written by generic stores, read by the tensor cores
  __syncthreads();
  // The scale s = 1 / (||X~_0||_F + eps) comes from the first Gram's diagonal:
  // ||X~_0||_F^2 = trace(X~_0 X~_0^T), the same exact bf16 products summed in
  // fp32, so the first product starts right after the load. Zero steps have
  // no Gram: sum the squares directly.
  float s = 1.0f;
  if (p.steps == 0) {
    float ss = 0.0f;
    for (int c = 8 * cq; c < npad; c += 32) {
      const uint4 q = *reinterpret_cast<const uint4*>(sX + soff(row, c));
      const uint32_t w4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float x0 = __uint_as_float(w4[k] << 16), x1 = __uint_as_float(w4[k] & 0xFFFF0000u);
        ss = fmaf(x0, x0, ss);
        ss = fmaf(x1, x1, ss);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) red[warp] = ss;
    __syncthreads();
    // fixed-order fp32 sum of the warp partials (FP64 arithmetic is slow on
    // this part, and every thread needs the scale)
    float tot = 0.0f;
#pragma unroll
    for (int w = 0; w < SM_WARPS; ++w) tot += red[w];
    s = 1.0f / (sqrtf(tot) + p.eps);
  }

  const uint32_t lane_base = tmem + (static_cast<uint32_t>(lq * 32) << 16);
  const uint32_t xs = smem_u32(sX), as = smem_u32(sA), bs = smem_u32(sB);
  constexpr uint32_t ID128 = idesc_make(1u, 128, 128, false, false);
  uint32_t ph = 0;
  bool ok = true;
  for (int step = 0; ok && step < p.steps; ++step) {
    // ---- A = X X^T (K = n)
    if (t == 0) {
      tc_fence_after();
      for (int kk = 0; kk < npad / 16; ++kk) {
        const uint32_t a = xs + (kk >> 2) * CHUNK + (kk & 3) * 32;
        mma_f16(tmem, sdesc_sw128(a, 16, 1024), sdesc_sw128(a, 16, 1024), ID128, kk > 0 ? 1u : 0u);
      }
      mma_commit(&bar[0]);
    }
    if (!(ok = wait_mma(&bar[0], ph, abort_flag, p.status))) break;
    ph ^= 1u;
    tc_fence_after();
    {
      const int c = 32 * cq;
      uint32_t v[32];
      tmem_ld32(lane_base + c, v);
      tmem_ld_wait();
      if (step == 0) {
        // the warp whose column chunk is its own row block holds the diagonal
        // A~[row][row] in register `lane`
        if (cq == lq) {
          float d = 0.0f;
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j == lane) d = __uint_as_float(v[j]);
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
          if (lane == 0) red[lq] = d;
        }
        __syncthreads();
        s = 1.0f / (sqrtf(red[0] + red[1] + red[2] + red[3]) + p.eps);
      }
      const float sc = step == 0 ? s : 1.0f;
      const float sc2 = sc * sc;
      {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          uint4 q;
          q.x = pack2(sc2 * __uint_as_float(v[8 * u + 0]), sc2 * __uint_as_float(v[8 * u + 1]));
          q.y = pack2(sc2 * __uint_as_float(v[8 * u + 2]), sc2 * __uint_as_float(v[8 * u + 3]));
          q.z = pack2(sc2 * __uint_as_float(v[8 * u + 4]), sc2 * __uint_as_float(v[8 * u + 5]));
          q.w = pack2(sc2 * __uint_as_float(v[8 * u + 6]), sc2 * __uint_as_float(v[8 * u + 7]));
          *reinterpret_cast<uint4*>(sA + soff(row, c + 8 * u)) = q;
        }
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    // ---- A*A (K = 128), accumulator in columns [128, 256)
    if (t == 0) {
      tc_fence_after();
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t a = as + (kk >> 2) * CHUNK + (kk & 3) * 32;
        mma_f16(tmem + 128, sdesc_sw128(a, 16, 1024), sdesc_sw128(a, 16, 1024), ID128, kk > 0 ? 1u : 0u);
      }
      mma_commit(&bar[0]);
    }
    if (!(ok = wait_mma(&bar[0], ph, abort_flag, p.status))) break;
    ph ^= 1u;
    tc_fence_after();
    {
      const int c = 32 * cq;
      uint32_t v[32];
      tmem_ld32(lane_base + 128 + c, v);
      tmem_ld_wait();
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint4 qa = *reinterpret_cast<const uint4*>(sA + soff(row, c + 8 * u));
        const uint32_t wa[4] = {qa.x, qa.y, qa.z, qa.w};
        uint32_t wb[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float a0 = __uint_as_float(wa[k] << 16), a1 = __uint_as_float(wa[k] & 0xFFFF0000u);
          wb[k] = pack2(p.b * a0 + p.c * __uint_as_float(v[8 * u + 2 * k]),
                        p.b * a1 + p.c * __uint_as_float(v[8 * u + 2 * k + 1]));
        }
        *reinterpret_cast<uint4*>(sB + soff(row, c + 8 * u)) = make_uint4(wb[0], wb[1], wb[2], wb[3]);
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    const float sc = step == 0 ? s : 1.0f;
    // ---- B*X (K = 128): B K-major, X MN-major; N in pieces of at most 256
    if (t == 0) {
      tc_fence_after();
      for (int nc = 0; nc < npad / 64; nc += 4) {
        const int N = min(256, npad - nc * 64);
        const uint32_t id = idesc_make(1u, 128, static_cast<uint32_t>(N), false, true);
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t a = bs + (kk >> 2) * CHUNK + (kk & 3) * 32;
          const uint32_t b = xs + nc * CHUNK + kk * (16 * 128);
          mma_f16(tmem + nc * 64, sdesc_sw128(a, 16, 1024), sdesc_sw128(b, CHUNK, 1024), id, kk > 0 ? 1u : 0u);
        }
      }
      mma_commit(&bar[0]);
    }
    if (!(ok = wait_mma(&bar[0], ph, abort_flag, p.status))) break;
    ph ^= 1u;
    tc_fence_after();
#pragma unroll 1
    for (int c0 = 32 * cq; c0 < npad; c0 += 256) {
      // this warp's chunks c0 and c0 + 128: both TMEM loads in flight at once
      const bool two = c0 + 128 < npad;
      uint32_t v2[2][32];
      tmem_ld32(lane_base + c0, v2[0]);
      if (two) tmem_ld32(lane_base + c0 + 128, v2[1]);
      tmem_ld_wait();
#pragma unroll
      for (int h = 0; h < 2; ++h) {
      if (h == 1 && !two) break;
      const int c = c0 + 128 * h;
      const uint32_t* v = v2[h];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        uint4* px = reinterpret_cast<uint4*>(sX + soff(row, c + 8 * u));
        const uint4 qx = *px;
        const uint32_t wx[4] = {qx.x, qx.y, qx.z, qx.w};
        uint32_t wo[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float x0 = __uint_as_float(wx[k] << 16), x1 = __uint_as_float(wx[k] & 0xFFFF0000u);
          wo[k] = pack2(sc * (p.a * x0 + __uint_as_float(v[8 * u + 2 * k])),
                        sc * (p.a * x1 + __uint_as_float(v[8 * u + 2 * k + 1])));
        }
        *px = make_uint4(wo[0], wo[1], wo[2], wo[3]);
      }
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
  }

  if (ok) {
    // ---- store: cropped, transposed back, bf16 (zero steps: s X~_0)
    const float so = p.steps == 0 ? s : 1.0f;
    for (int r = warp; r < M.rows; r += SM_THREADS / 32) {
      unsigned short* dst = out_row(p, M, r);
      for (int c0 = lane * 8; c0 < M.cols; c0 += 32 * 8) {
        unsigned short v[8];
        if (!tr) {
          // row r of X: the 8 elements are one 16-byte unit of the swizzled row
          *reinterpret_cast<uint4*>(v) = *reinterpret_cast<const uint4*>(sX + soff(r, c0));
        } else {
#pragma unroll
          for (int k = 0; k < 8; ++k)
            v[k] = *reinterpret_cast<const unsigned short*>(sX + soff(min(c0 + k, M.cols - 1), r));
        }
        if (p.steps == 0) {
#pragma unroll
          for (int k = 0; k < 8; k += 2) {
            const uint32_t w = pack2(so * bf(v[k]), so * bf(v[k + 1]));
            v[k] = static_cast<unsigned short>(w & 0xFFFFu);
            v[k + 1] = static_cast<unsigned short>(w >> 16);
          }
        }
        if (c0 + 8 <= M.cols && (reinterpret_cast<uintptr_t>(dst + c0) & 15) == 0) {
          *reinterpret_cast<uint4*>(dst + c0) = *reinterpret_cast<const uint4*>(v);
        } else {
#pragma unroll
          for (int k = 0; k < 8; ++k)
            if (c0 + k < M.cols) dst[c0 + k] = v[k];
        }
      }
    }
  } else if (t == 0) {
    // a wait gave up: let any MMA still in flight finish before TMEM is freed
    mma_commit(&bar[1]);
    mbar_wait_drain(&bar[1], 0, p.status);
  }
  (void)m;
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, tmem_cols);
  }
}

// The kernel with a table of N matrices; the function attribute (shared
// memory above 48 KB) is set once per device.
template <int N>
cudaError_t launch_small_n(const SmallParams& p, size_t smem, cudaStream_t st) {
  static std::atomic<unsigned long long> attr_set{0};
  auto kern = ns_small_kernel<SmallParamsT<N>>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(attr_set.load() & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(small_smem_bytes(SMALL_MAX_N)));
    if (e != cudaSuccess) return e;
    attr_set.fetch_or(bit);
  }
  if constexpr (N == SMALL_MAX_MATS) {
    e = launch_pdl(kern, dim3(static_cast<unsigned>(p.count)), dim3(SM_THREADS), smem, st, p);
  } else {
    SmallParamsT<N> q;
    std::memcpy(&q, &p, offsetof(SmallParams, mat));
    std::memcpy(q.mat, p.mat, sizeof(SmallMat) * static_cast<size_t>(p.count));
    e = launch_pdl(kern, dim3(static_cast<unsigned>(p.count)), dim3(SM_THREADS), smem, st, q);
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_small(const SmallParams& p, cudaStream_t st) {
  if (p.count <= 0) return cudaSuccess;
  if (p.count > SMALL_MAX_MATS) return cudaErrorInvalidValue;
  if (p.n_pad < 64 || p.n_pad > SMALL_MAX_N || p.n_pad % 64) return cudaErrorInvalidValue;
  const size_t smem = small_smem_bytes(p.n_pad);
  if (p.count <= 16) return launch_small_n<16>(p, smem, st);
  if (p.count <= 64) return launch_small_n<64>(p, smem, st);
  return launch_small_n<SMALL_MAX_MATS>(p, smem, st);
}

}  // namespace nsk
