// Memory-bound kernels around the Newton-Schulz products (Megatron-Core API
// page owner_planning, ns_cost_fn: view as (shape[0], prod(shape[1:])),
// normalise, transpose so rows <= cols; the result is transposed back).
//
//   ns_prep_kernel    bf16 path: X~_0 = T or T^T, zero-padded to m_pad x n_pad,
//                     unscaled, and per-block partial sums of squares (one pass)
//   ns_sumsq_kernel   fp32 paths: partial sums of squares over 32K-element chunks
//   ns_scale_kernel   scale = 1 / (sqrt(sum of partials) + eps), fixed order
//   ns_store_kernel   out = X_k (or X_k^T) cropped to the tensor's (rows, cols)
//
// Each launch covers up to PRO_MAX_MATS matrices of one shape bucket; the
// per-matrix pointers travel in the parameter block.
#include <cuda_bf16.h>

#include "kernels.h"
#include "launch.cuh"
#include "ptx.cuh"
#include "status.h"

namespace nsk {
namespace {

constexpr int SUMSQ_THREADS = 256;
constexpr long long SUMSQ_CHUNK = 32768;
constexpr int TILE = 64;

__device__ __forceinline__ float bf16_to_f(unsigned short h) { return __uint_as_float(uint32_t(h) << 16); }

__device__ __forceinline__ float block_sum(float v) {
  __shared__ float red[32];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int w = threadIdx.x / 32, l = threadIdx.x % 32;
  if (l == 0) red[w] = v;
  __syncthreads();
  v = (threadIdx.x < blockDim.x / 32) ? red[threadIdx.x] : 0.0f;
  if (w == 0) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  }
  return v;
}

__global__ void __launch_bounds__(SUMSQ_THREADS) ns_sumsq_kernel(const __grid_constant__ ProParams p) {
  nsptx::griddep_wait();
  nsptx::griddep_launch_dependents();
  const MatDesc& d = p.md[blockIdx.y];
  const long long c0 = static_cast<long long>(blockIdx.x) * SUMSQ_CHUNK;
  if (c0 >= d.numel) return;
  const long long c1 = min(d.numel, c0 + SUMSQ_CHUNK);
  const unsigned short* src = reinterpret_cast<const unsigned short*>(d.in);
  float acc = 0.0f;
  if ((reinterpret_cast<uintptr_t>(src) & 15) == 0) {
    const long long v0 = c0 / 8, v1 = c1 / 8;  // c0 is a multiple of 8
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    for (long long i = v0 + threadIdx.x; i < v1; i += blockDim.x) {
      const uint4 q = __ldg(&s4[i]);
      const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float lo = __uint_as_float(w[k] << 16), hi = __uint_as_float(w[k] & 0xFFFF0000u);
        acc = fmaf(lo, lo, acc);
        acc = fmaf(hi, hi, acc);
      }
    }
    for (long long i = v1 * 8 + threadIdx.x; i < c1; i += blockDim.x) {
      const float x = bf16_to_f(src[i]);
      acc = fmaf(x, x, acc);
    }
  } else {
    for (long long i = c0 + threadIdx.x; i < c1; i += blockDim.x) {
      const float x = bf16_to_f(src[i]);
      acc = fmaf(x, x, acc);
    }
  }
  acc = block_sum(acc);
  if (threadIdx.x == 0) d.partial[blockIdx.x] = acc;
}

__global__ void __launch_bounds__(256) ns_scale_kernel(const __grid_constant__ ProParams p) {
  nsptx::griddep_wait();
  nsptx::griddep_launch_dependents();
  const MatDesc& d = p.md[blockIdx.x];
  double s = 0.0;
  for (int i = threadIdx.x; i < p.nchunks; i += blockDim.x) s += static_cast<double>(d.partial[i]);
  // fixed-order reduction in double
  __shared__ double red[256];
  red[threadIdx.x] = s;
  __syncthreads();
  for (int o = blockDim.x / 2; o > 0; o >>= 1) {
    if (threadIdx.x < o) red[threadIdx.x] += red[threadIdx.x + o];
    __syncthreads();
  }
  if (threadIdx.x == 0) *d.scale = static_cast<float>(1.0 / (sqrt(red[0]) + static_cast<double>(p.eps)));
}

__device__ __forceinline__ float sq8(const uint4& q) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
  float acc = 0.0f;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float lo = __uint_as_float(w[k] << 16), hi = __uint_as_float(w[k] & 0xFFFF0000u);
    acc = fmaf(lo, lo, acc);
    acc = fmaf(hi, hi, acc);
  }
  return acc;
}

// bf16 prologue, one pass: V = T (rows <= cols) or T^T copied unscaled into
// X~_0 (m_pad x n_pad, zero padded) and the sum of squares of each 64-row
// block of V written to partial[block]. The scale 1 / (||T||_F + eps) is
// applied by the first step's products (A = s^2 X~ X~^T, X_1 = s (a X~ + B X~)),
// which equals running the step on X_0 = s X~. The input is bf16, so X~_0
// holds it exactly. blockIdx.x = block of 64 rows x 1024 columns of X~_0
// (row-stripe major), blockIdx.y = matrix; small batches still fill the GPU.
//
// Plain: 16-byte vectors of T rows to X~_0 rows, four loads in flight per
// thread. Transposed: the block is 64 columns of T, walked in 64 x 64 tiles
// (64 rows of T x 128 bytes in, 64 rows of X~_0 x 128 bytes out, both whole
// lines per warp access) through a double-buffered bf16 tile in shared memory
// (rows of 33 words: conflict-free writes, 2-way reads).
constexpr int PREP_THREADS = 256;
constexpr int PREP_COLS = 1024;  // X~_0 columns per CTA (a multiple of 64)

__global__ void __launch_bounds__(PREP_THREADS) ns_prep_kernel(const __grid_constant__ ProParams p) {
  nsptx::griddep_wait();
  nsptx::griddep_launch_dependents();
  const MatDesc& d = p.md[blockIdx.y];
  const unsigned short* __restrict__ src = reinterpret_cast<const unsigned short*>(d.in);
  uint4* __restrict__ x4 = reinterpret_cast<uint4*>(d.x);
  // row j of the input tensor (d.cols elements): contiguous in its home
  // buffer, or in the rank buffer holding its row shard
  const long long row_len = d.cols;
  auto trow = [&](long long j) -> const unsigned short* {
    if (!p.from_ranks) return src + j * row_len;
    const int r = static_cast<int>(j / d.shard_rows);
    return reinterpret_cast<const unsigned short*>(p.rank_ptr[r]) + d.rank_off + (j - static_cast<long long>(r) * d.shard_rows) * row_len;
  };
  const bool base_aligned = p.from_ranks ? (p.ranks_aligned && d.rank_off % 8 == 0)
                                         : (reinterpret_cast<uintptr_t>(src) & 15) == 0;
  const int nv = p.n_pad / 8;  // 16-byte vectors per X~_0 row
  // this CTA: rows [i0, i0 + 64) of X~_0, columns [c0, c1) (a block of
  // PREP_COLS, the last one shorter)
  const int ncb = (p.n_pad + PREP_COLS - 1) / PREP_COLS;
  const int i0 = (blockIdx.x / ncb) * TILE;
  const int c0 = (blockIdx.x % ncb) * PREP_COLS, c1 = min(p.n_pad, c0 + PREP_COLS);
  float acc = 0.0f;
  if (!d.transposed) {
    const bool vec = (p.n % 8 == 0) && base_aligned;
    const int nvb = (c1 - c0) / 8;  // vectors of a row in this column block
    const int total = TILE * nvb;
    constexpr int U = 4;
    for (int base = threadIdx.x; base < total; base += U * PREP_THREADS) {
      uint4 q[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = base + u * PREP_THREADS;
        const int i = i0 + v / nvb, j0 = c0 + (v % nvb) * 8;
        q[u] = make_uint4(0, 0, 0, 0);
        if (v < total && i < p.m) {
          const unsigned short* row = trow(i);
          if (vec && j0 + 8 <= p.n) {
            q[u] = __ldg(reinterpret_cast<const uint4*>(row + j0));
          } else if (j0 < p.n) {
            uint16_t h[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) h[k] = j0 + k < p.n ? row[j0 + k] : 0;
            q[u] = make_uint4(h[0] | (uint32_t(h[1]) << 16), h[2] | (uint32_t(h[3]) << 16),
                              h[4] | (uint32_t(h[5]) << 16), h[6] | (uint32_t(h[7]) << 16));
          }
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int v = base + u * PREP_THREADS;
        if (v < total) {
          acc += sq8(q[u]);
          x4[static_cast<long long>(i0 + v / nvb) * nv + c0 / 8 + v % nvb] = q[u];
        }
      }
    }
  } else {
    // X~[i][j] = T[j][i], T row-major n x m (rows j, cols i)
    __shared__ uint32_t tile[2][TILE][TILE / 2 + 1];
    const bool vec = (p.m % 8 == 0) && base_aligned;
    const int jt0 = c0 / TILE, jt1 = c1 / TILE;  // X~_0 column tiles = T row tiles
    // each thread moves two 16-byte vectors per tile: vector q = threadIdx.x + 256 h
    auto load = [&](int jt, uint4 (&r)[2]) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int q = threadIdx.x + h * PREP_THREADS;
        const int j = jt * TILE + q / 8, i = i0 + (q % 8) * 8;
        r[h] = make_uint4(0, 0, 0, 0);
        if (j < p.n && i < p.m) {
          const unsigned short* row = trow(j);
          if (vec && i + 8 <= p.m) {
            r[h] = __ldg(reinterpret_cast<const uint4*>(row + i));
          } else {
            uint16_t e[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) e[k] = i + k < p.m ? row[i + k] : 0;
            r[h] = make_uint4(e[0] | (uint32_t(e[1]) << 16), e[2] | (uint32_t(e[3]) << 16),
                              e[4] | (uint32_t(e[5]) << 16), e[6] | (uint32_t(e[7]) << 16));
          }
        }
      }
    };
    uint4 r[2];
    load(jt0, r);
    for (int jt = jt0; jt < jt1; ++jt) {
      const int buf = jt & 1;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int q = threadIdx.x + h * PREP_THREADS;
        const int jj = q / 8, iw = (q % 8) * 4;  // row jj of the tile, word iw (= column 2 iw)
        acc += sq8(r[h]);
        tile[buf][jj][iw] = r[h].x;
        tile[buf][jj][iw + 1] = r[h].y;
        tile[buf][jj][iw + 2] = r[h].z;
        tile[buf][jj][iw + 3] = r[h].w;
      }
      __syncthreads();
      if (jt + 1 < jt1) load(jt + 1, r);  // next tile's loads overlap this tile's stores
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int q = threadIdx.x + h * PREP_THREADS;
        const int ii = q / 8, jv = (q % 8) * 8;  // row ii of X~_0's tile, columns jv..jv+7
        const unsigned short* t16 = reinterpret_cast<const unsigned short*>(&tile[buf][0][0]);
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t lo = t16[(jv + 2 * k) * (TILE + 2) + ii];
          const uint32_t hi = t16[(jv + 2 * k + 1) * (TILE + 2) + ii];
          w[k] = lo | (hi << 16);
        }
        x4[(static_cast<long long>(i0 + ii) * p.n_pad + jt * TILE + jv) / 8] = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
  }
  acc = block_sum(acc);
  if (threadIdx.x == 0) d.partial[blockIdx.x] = acc;
}

// One 64 x 64 tile of the output (rows x cols) per CTA.
__global__ void __launch_bounds__(256) ns_store_kernel(const __grid_constant__ ProParams p) {
  nsptx::griddep_wait();
  nsptx::griddep_launch_dependents();
  __shared__ float tile[TILE][TILE + 1];
  const MatDesc& d = p.md[blockIdx.y];
  const int rows = d.rows, cols = d.cols;
  const int tiles_c = (cols + TILE - 1) / TILE;
  const int ti = blockIdx.x / tiles_c, tj = blockIdx.x % tiles_c;
  const int i0 = ti * TILE, j0 = tj * TILE;
  const unsigned short* x = reinterpret_cast<const unsigned short*>(d.xfinal);
  const float sc = p.apply_scale ? *d.scale : 1.0f;  // zero steps: X~_0 is stored unscaled
  const int tx = threadIdx.x % TILE, ty = threadIdx.x / TILE;
  if (!d.transposed) {
    for (int ii = ty; ii < TILE; ii += 4) {
      const int i = i0 + ii, j = j0 + tx;
      if (i < rows && j < cols) {
        const float v = sc * bf16_to_f(x[static_cast<long long>(i) * p.n_pad + j]);
        if (p.out_f32)
          reinterpret_cast<float*>(d.out)[static_cast<long long>(i) * cols + j] = v;
        else
          reinterpret_cast<__nv_bfloat16*>(d.out)[static_cast<long long>(i) * cols + j] = __float2bfloat16_rn(v);
      }
    }
  } else {
    // out[i][j] = X[j][i]; X is m_pad x n_pad with j < m (= cols), i < n (= rows)
    for (int jj = ty; jj < TILE; jj += 4) {
      const int j = j0 + jj, i = i0 + tx;
      float v = 0.0f;
      if (i < rows && j < cols) v = sc * bf16_to_f(x[static_cast<long long>(j) * p.n_pad + i]);
      tile[jj][tx] = v;
    }
    __syncthreads();
    for (int ii = ty; ii < TILE; ii += 4) {
      const int i = i0 + ii, j = j0 + tx;
      if (i < rows && j < cols) {
        const float v = tile[tx][ii];
        if (p.out_f32)
          reinterpret_cast<float*>(d.out)[static_cast<long long>(i) * cols + j] = v;
        else
          reinterpret_cast<__nv_bfloat16*>(d.out)[static_cast<long long>(i) * cols + j] = __float2bfloat16_rn(v);
      }
    }
  }
}

__device__ __forceinline__ float tf32_round(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return __uint_as_float(r);
}

// fp32-Gram prologue: one 64 x 64 tile of X_0 = scale * V per CTA, written as
// hi/lo TF32 pairs both as X (m_pad x n_pad) and as X^T (n_pad x m_pad).
__global__ void __launch_bounds__(256) ns_prep32_kernel(const __grid_constant__ ProParams p) {
  nsptx::griddep_wait();
  nsptx::griddep_launch_dependents();
  __shared__ float tile[TILE][TILE + 1];
  const MatDesc& d = p.md[blockIdx.y];
  const float s = *d.scale;
  const unsigned short* src = reinterpret_cast<const unsigned short*>(d.in);
  float* xh = reinterpret_cast<float*>(d.x);
  float* xl = xh + p.x_split;
  float* th = xh + 2 * p.x_split;
  float* tl = xh + 3 * p.x_split;
  const int tiles_n = p.n_pad / TILE;
  const int ti = blockIdx.x / tiles_n, tj = blockIdx.x % tiles_n;
  const int i0 = ti * TILE, j0 = tj * TILE;
  const int tx = threadIdx.x % TILE, ty = threadIdx.x / TILE;
  if (!d.transposed) {
    for (int ii = ty; ii < TILE; ii += 4) {   // V[i][j] = T[i][j], coalesced along j
      const int i = i0 + ii, j = j0 + tx;
      tile[ii][tx] = (i < p.m && j < p.n) ? s * bf16_to_f(src[static_cast<long long>(i) * p.n + j]) : 0.0f;
    }
  } else {
    for (int jj = ty; jj < TILE; jj += 4) {   // V[i][j] = T[j][i], coalesced along i
      const int j = j0 + jj, i = i0 + tx;
      tile[tx][jj] = (i < p.m && j < p.n) ? s * bf16_to_f(src[static_cast<long long>(j) * p.m + i]) : 0.0f;
    }
  }
  __syncthreads();
  for (int ii = ty; ii < TILE; ii += 4) {     // X rows
    const float v = tile[ii][tx], h = tf32_round(v);
    const long long e = static_cast<long long>(i0 + ii) * p.n_pad + j0 + tx;
    xh[e] = h;
    xl[e] = v - h;
  }
  for (int jj = ty; jj < TILE; jj += 4) {     // X^T rows
    const float v = tile[tx][jj], h = tf32_round(v);
    const long long e = static_cast<long long>(j0 + jj) * p.m_pad + i0 + tx;
    th[e] = h;
    tl[e] = v - h;
  }
}

// fp32-Gram store (used when the last B*X launch could not store directly):
// out (rows x cols, fp32) from X_k = hi + lo.
__global__ void __launch_bounds__(256) ns_store32_kernel(const __grid_constant__ ProParams p) {
  nsptx::griddep_wait();
  nsptx::griddep_launch_dependents();
  __shared__ float tile[TILE][TILE + 1];
  const MatDesc& d = p.md[blockIdx.y];
  const int rows = d.rows, cols = d.cols;
  const int tiles_c = (cols + TILE - 1) / TILE;
  const int ti = blockIdx.x / tiles_c, tj = blockIdx.x % tiles_c;
  const int i0 = ti * TILE, j0 = tj * TILE;
  const float* xh = reinterpret_cast<const float*>(d.xfinal);
  const float* xl = xh + p.x_split;
  float* out = reinterpret_cast<float*>(d.out);
  const int tx = threadIdx.x % TILE, ty = threadIdx.x / TILE;
  if (!d.transposed) {
    for (int ii = ty; ii < TILE; ii += 4) {
      const int i = i0 + ii, j = j0 + tx;
      if (i < rows && j < cols) {
        const long long e = static_cast<long long>(i) * p.n_pad + j;
        out[static_cast<long long>(i) * cols + j] = xh[e] + xl[e];
      }
    }
  } else {
    for (int jj = ty; jj < TILE; jj += 4) {
      const int j = j0 + jj, i = i0 + tx;
      float v = 0.0f;
      if (i < rows && j < cols) {
        const long long e = static_cast<long long>(j) * p.n_pad + i;
        v = xh[e] + xl[e];
      }
      tile[jj][tx] = v;
    }
    __syncthreads();
    for (int ii = ty; ii < TILE; ii += 4) {
      const int i = i0 + ii, j = j0 + tx;
      if (i < rows && j < cols) out[static_cast<long long>(i) * cols + j] = tile[tx][ii];
    }
  }
}

}  // namespace

cudaError_t launch_prep32(const ProParams& p, cudaStream_t st) {
  if (p.count <= 0) return cudaSuccess;
  const int tiles = (p.m_pad / TILE) * (p.n_pad / TILE);
  {
    const cudaError_t e = launch_pdl(ns_prep32_kernel, dim3(tiles, p.count), dim3(256), 0, st, p);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

cudaError_t launch_store32(const ProParams& p, cudaStream_t st) {
  if (p.count <= 0) return cudaSuccess;
  const int rows = p.md[0].rows, cols = p.md[0].cols;
  const int tiles = ((rows + TILE - 1) / TILE) * ((cols + TILE - 1) / TILE);
  {
    const cudaError_t e = launch_pdl(ns_store32_kernel, dim3(tiles, p.count), dim3(256), 0, st, p);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

cudaError_t launch_sumsq(const ProParams& p, cudaStream_t st) {
  if (p.count <= 0 || p.nchunks <= 0) return cudaSuccess;
  {
    const cudaError_t e = launch_pdl(ns_sumsq_kernel, dim3(p.nchunks, p.count), dim3(SUMSQ_THREADS), 0, st, p);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

cudaError_t launch_scale(const ProParams& p, cudaStream_t st) {
  if (p.count <= 0) return cudaSuccess;
  {
    const cudaError_t e = launch_pdl(ns_scale_kernel, dim3(p.count), dim3(256), 0, st, p);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

cudaError_t launch_prep(const ProParams& p, cudaStream_t st) {
  if (p.count <= 0) return cudaSuccess;
  // one CTA per 64-row stripe and 1024-column block of X~_0 (p.nchunks of
  // them per matrix, each writing one partial sum of squares)
  const int ncb = (p.n_pad + PREP_COLS - 1) / PREP_COLS;
  if (p.nchunks != (p.m_pad / TILE) * ncb) return cudaErrorInvalidValue;
  {
    const cudaError_t e = launch_pdl(ns_prep_kernel, dim3(p.nchunks, p.count), dim3(PREP_THREADS), 0, st, p);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

cudaError_t launch_store(const ProParams& p, cudaStream_t st) {
  if (p.count <= 0) return cudaSuccess;
  const int rows = p.md[0].rows, cols = p.md[0].cols;
  // all matrices of a bucket have the same (rows, cols) up to a transpose,
  // so the tile count is the same for each
  const int tiles = ((rows + TILE - 1) / TILE) * ((cols + TILE - 1) / TILE);
  {
    const cudaError_t e = launch_pdl(ns_store_kernel, dim3(tiles, p.count), dim3(256), 0, st, p);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

}  // namespace nsk
