// fp32-Gram variant of the three Newton-Schulz products (Megatron-Core API page
// owner_planning, ns_cost_fn; Megatron-LM issue #6720 pairs an fp32/TF32 Gram
// with a trace ridge to harden the iteration):
//
//   PH32_GRAM  A  = X X^T                 symmetric: upper tiles + mirror
//   PH32_A2B   B  = b A + c (A A)         symmetric: upper tiles + mirror
//   PH32_BXT   X' = a X + B X, computed as (B X)^T = X^T B (B symmetric)
//
// Every matrix is held in fp32 as a pair (hi, lo): hi = x rounded to TF32,
// lo = x - hi. Each product is accumulated in fp32 TMEM from three TF32
// tensor-core products hi*hi + hi*lo + lo*hi (the split-precision scheme of
// Markidis et al. 2018 and Ootomo & Yokota 2022), which keeps fp32-level
// accuracy; the dropped lo*lo term is ~2^-22 relative.
//
// All operands are K-major (K blocks of 16 fp32: rows of 64 bytes, 64-byte
// swizzle; four 48 KB stages):
// X is kept both as X (m_pad x n_pad, for the Gram) and X^T (n_pad x m_pad,
// for B*X), and the B*X epilogue writes both copies of the next X.
// Structure as in gemm.cu: persistent CTAs, a TMA producer thread, one MMA
// issuing thread (tcgen05.mma.cta_group::1.kind::tf32, M=128, N=256, K=8),
// two TMEM accumulators, four epilogue warps; every wait is bounded.
#include <algorithm>

#include "kernels.h"
#include "launch.cuh"
#include "ptx.cuh"

namespace nsk {
namespace {

using namespace nsptx;

constexpr int BM = 128, BN = 256, BK = GEMM32_BK, UK = 8;
constexpr int STAGES = 4;
constexpr uint32_t A_BYTES = BM * BK * 4;  // 8 KB
constexpr uint32_t B_BYTES = BN * BK * 4;  // 16 KB
constexpr uint32_t STAGE_BYTES = 2 * A_BYTES + 2 * B_BYTES;  // hi and lo of both operands
constexpr uint32_t TMEM_COLS = 2 * BN;
constexpr int THREADS = 192;
constexpr size_t SMEM_BYTES = 1024 + size_t(STAGES) * STAGE_BYTES + 256;

__device__ __forceinline__ float tf32_round(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return __uint_as_float(r);
}

template <int PHASE, typename P>
__device__ __forceinline__ void decode_tile32(const P& p, long long t, int& b, int& mat, int& tm, int& tn) {
  b = 0;
  while (b + 1 < p.nb && t >= p.bk[b + 1].tile_begin) ++b;
  const Gemm32Bucket& B = p.bk[b];
  const long long local = t - B.tile_begin;
  mat = static_cast<int>(local / B.tiles_per_mat);
  int r = static_cast<int>(local % B.tiles_per_mat);
  if (PHASE == PH32_BXT) {
    tm = r / B.tiles_n;
    tn = r % B.tiles_n;
  } else {
    tm = 0;
    while (true) {
      const int tn0 = (tm * BM) / BN;
      const int cnt = B.tiles_n - tn0;
      if (r < cnt) {
        tn = tn0 + r;
        break;
      }
      r -= cnt;
      ++tm;
    }
  }
}

// Epilogue of one tile for the warp owning accumulator rows [32 lg, +32):
// TMEM accumulator `acc` (256 fp32 columns) -> the phase's outputs. Shared by
// the 1-SM and the 2-SM kernel (in the latter each CTA holds its own 128 rows).
template <int PHASE, bool FINAL, typename P>
__device__ __forceinline__ void epilogue32_tile(const P& p, int b, int mat, int tm, int tn, uint32_t tmem_base,
                                                uint32_t acc, int lg, int lane) {
  constexpr bool SYRK = (PHASE != PH32_BXT);
  const Gemm32Bucket& B = p.bk[b];
  // the second row block of a pair past the last tile row stores nothing
  if (tm >= B.tiles_m) return;
  const int r0w = tm * BM + lg * 32;
  const int r = r0w + lane;  // Gram/A2B: row of A/B; BXT: column j of X (n index)
  const long long mo = static_cast<long long>(mat) * B.mat_stride;
  const long long mt = static_cast<long long>(mat) * B.mat_stride_t;
#pragma unroll 1
  for (int c0 = 0; c0 < BN; c0 += 32) {
    const int cg = tn * BN + c0;
    if (cg >= B.cols_valid) break;
    if (SYRK && cg + 31 < r0w) continue;
    uint32_t v[32];
    tmem_ld32(tmem_base + (static_cast<uint32_t>(lg * 32) << 16) + acc * BN + c0, v);
    tmem_ld_wait();
    float f[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) f[j] = __uint_as_float(v[j]);
    if (PHASE == PH32_A2B) {
      // out = delta*I + beta*aux + gamma*(L R); aux = hi + lo (standard
      // step: B = b*A + c*(A A); Gram-space steps: Q, Q*A, Q*T, Q*P)
      float dl = B.delta, be = B.beta, ga = B.gamma;
      if (B.coef) {
        dl = B.coef[3 * mat];
        be = B.coef[3 * mat + 1];
        ga = B.coef[3 * mat + 2];
      }
#pragma unroll
      for (int j = 0; j < 32; ++j) f[j] *= ga;
      if (B.aux_h) {
        const float4* h4 = reinterpret_cast<const float4*>(B.aux_h + mo + static_cast<long long>(r) * B.ld + cg);
        const float4* l4 = reinterpret_cast<const float4*>(B.aux_l + mo + static_cast<long long>(r) * B.ld + cg);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float4 h = h4[q], l = l4[q];
          f[4 * q + 0] += be * (h.x + l.x);
          f[4 * q + 1] += be * (h.y + l.y);
          f[4 * q + 2] += be * (h.z + l.z);
          f[4 * q + 3] += be * (h.w + l.w);
        }
      }
      if (r >= cg && r < cg + 32) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (cg + j == r) f[j] += dl;
      }
    }
    if (SYRK) {
      float fh[32], fl[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        fh[j] = tf32_round(f[j]);
        fl[j] = f[j] - fh[j];
      }
      float* oh = B.out_h + mo + static_cast<long long>(r) * B.ld + cg;
      float* ol = B.out_l + mo + static_cast<long long>(r) * B.ld + cg;
      if (cg >= r) {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          reinterpret_cast<float4*>(oh)[q] = make_float4(fh[4 * q], fh[4 * q + 1], fh[4 * q + 2], fh[4 * q + 3]);
          reinterpret_cast<float4*>(ol)[q] = make_float4(fl[4 * q], fl[4 * q + 1], fl[4 * q + 2], fl[4 * q + 3]);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (cg + j >= r) {
            oh[j] = fh[j];
            ol[j] = fl[j];
          }
      }
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int c = cg + j;
        if (c > r) {
          B.out_h[mo + static_cast<long long>(c) * B.ld + r] = fh[j];
          B.out_l[mo + static_cast<long long>(c) * B.ld + r] = fl[j];
        }
      }
    } else {
      // acc[r][c] = (B X)[c][r]: c = m index (cg + j), r = n index.
      // X'[c][r] = a * X[c][r] + acc; X = hi + lo, read column-wise (lanes
      // hold consecutive r, so each access is contiguous across the warp).
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const long long e = mo + static_cast<long long>(cg + j) * B.ld + r;
        f[j] = p.alpha * (B.aux_h[e] + B.aux_l[e]) + f[j];
      }
      if constexpr (FINAL) {
        if (r < B.n_valid) {
          const unsigned long long ent = p.out_tab[B.out_first + mat];
          float* o = reinterpret_cast<float*>(ent & ~1ull);
          if (!(ent & 1ull)) {
            // output rows x cols = m x n: element (c, r)
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (cg + j < B.m_valid) o[static_cast<long long>(cg + j) * B.n_valid + r] = f[j];
          } else {
            // transposed tensor: output n x m, element (r, c), contiguous per thread
            float* dst = o + static_cast<long long>(r) * B.m_valid + cg;
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (cg + j < B.m_valid) dst[j] = f[j];
          }
        }
      } else {
        float fh[32], fl[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          fh[j] = tf32_round(f[j]);
          fl[j] = f[j] - fh[j];
        }
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const long long e = mo + static_cast<long long>(cg + j) * B.ld + r;
          B.out_h[e] = fh[j];
          B.out_l[e] = fl[j];
        }
        float* th = B.out_th + mt + static_cast<long long>(r) * B.ld_t + cg;
        float* tl = B.out_tl + mt + static_cast<long long>(r) * B.ld_t + cg;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          reinterpret_cast<float4*>(th)[q] = make_float4(fh[4 * q], fh[4 * q + 1], fh[4 * q + 2], fh[4 * q + 3]);
          reinterpret_cast<float4*>(tl)[q] = make_float4(fl[4 * q], fl[4 * q + 1], fl[4 * q + 2], fl[4 * q + 3]);
        }
      }
    }
  }
}

template <int PHASE, bool FINAL, typename P>
__global__ void __launch_bounds__(THREADS, 1) ns_gemm32_kernel(const __grid_constant__ P p) {
  static_assert(!FINAL || PHASE == PH32_BXT, "only the B*X phase has a final-store form");
  constexpr uint32_t IDESC = idesc_make(2u, BM, BN, false, false);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // stage s: [A hi | A lo | B hi | B lo]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  if (blockDim.x != THREADS) {
    if (threadIdx.x == 0) atomicOr(p.status, NS_DEV_BAD_LAUNCH);
    return;
  }
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    for (int b = 0; b < p.nb; ++b) {
      prefetch_tmap(&p.tmah[b]);
      prefetch_tmap(&p.tmal[b]);
      prefetch_tmap(&p.tmbh[b]);
      prefetch_tmap(&p.tmbl[b]);
    }
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // everything above is set-up; the data path starts after the predecessor
  griddep_wait();
  griddep_launch_dependents();

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer
    uint32_t stage = 0, phase = 0;
    long long issued = 0;
    for (long long t = blockIdx.x; t < p.total_tiles; t += gridDim.x) {
      int b, mat, tm, tn;
      decode_tile32<PHASE>(p, t, b, mat, tm, tn);
      const int kb_n = p.bk[b].k_blocks;
      for (int kb = 0; kb < kb_n; ++kb) {
        if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.status)) goto producer_done;
        mbar_arrive_expect_tx(&full[stage], STAGE_BYTES);
        uint8_t* base = smem + stage * STAGE_BYTES;
        tma_load_3d(base, &p.tmah[b], &full[stage], kb * BK, tm * BM, mat);
        tma_load_3d(base + A_BYTES, &p.tmal[b], &full[stage], kb * BK, tm * BM, mat);
        uint8_t* bh = base + 2 * A_BYTES;
        uint8_t* bl = bh + B_BYTES;
        tma_load_3d(bh, &p.tmbh[b], &full[stage], kb * BK, tn * BN, mat);
        tma_load_3d(bh + 128 * BK * 4, &p.tmbh[b], &full[stage], kb * BK, tn * BN + 128, mat);
        tma_load_3d(bl, &p.tmbl[b], &full[stage], kb * BK, tn * BN, mat);
        tma_load_3d(bl + 128 * BK * 4, &p.tmbl[b], &full[stage], kb * BK, tn * BN + 128, mat);
        ++issued;
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  producer_done:
    if (*abort_flag) {
      const long long first = issued > STAGES ? issued - STAGES : 0;
      for (long long i = first; i < issued; ++i)
        mbar_wait_drain(&full[i % STAGES], static_cast<uint32_t>((i / STAGES) & 1), p.status);
    }
  } else if (warp == 1 && lane == 0) {
    // ----------------------------------------------------------- MMA issuer
    uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
    for (long long t = blockIdx.x; t < p.total_tiles; t += gridDim.x) {
      int b, mat, tm, tn;
      decode_tile32<PHASE>(p, t, b, mat, tm, tn);
      const int kb_n = p.bk[b].k_blocks;
      if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag, p.status)) goto mma_done;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * BN;
      for (int kb = 0; kb < kb_n; ++kb) {
        if (!mbar_wait(&full[stage], phase, abort_flag, p.status)) goto mma_done;
        tc_fence_after();
        const uint32_t ah = smem_u32(smem + stage * STAGE_BYTES);
        const uint32_t al = ah + A_BYTES;
        const uint32_t bh = ah + 2 * A_BYTES;
        const uint32_t bl = bh + B_BYTES;
#pragma unroll
        for (int k = 0; k < BK / UK; ++k) {
          const uint32_t o = k * (UK * 4);  // 32 bytes per K step inside the 64-byte row
          const uint32_t first = (kb | k) != 0 ? 1u : 0u;
          mma_tf32(d_tmem, sdesc_sw64(ah + o, 16, 512), sdesc_sw64(bh + o, 16, 512), IDESC, first);
          mma_tf32(d_tmem, sdesc_sw64(ah + o, 16, 512), sdesc_sw64(bl + o, 16, 512), IDESC, 1u);
          mma_tf32(d_tmem, sdesc_sw64(al + o, 16, 512), sdesc_sw64(bh + o, 16, 512), IDESC, 1u);
        }
        mma_commit(&empty[stage]);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      mma_commit(&tfull[acc]);
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
  mma_done:
    if (*abort_flag) {
      mma_commit(drain);
      mbar_wait_drain(drain, 0, p.status);
    }
  } else if (warp >= 2) {
    // -------------------------------------------------------------- epilogue
    const int lg = warp & 3;
    uint32_t acc = 0, acc_phase = 0;
    for (long long t = blockIdx.x; t < p.total_tiles; t += gridDim.x) {
      int b, mat, tm, tn;
      decode_tile32<PHASE>(p, t, b, mat, tm, tn);
      if (!mbar_wait(&tfull[acc], acc_phase, abort_flag, p.status)) break;
      tc_fence_after();
      epilogue32_tile<PHASE, FINAL>(p, b, mat, tm, tn, tmem_base, acc, lg, lane);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// 2-SM form: a cluster of two CTAs computes a 256 x 256 tile with
// tcgen05.mma.cta_group::2.kind::tf32 (M = 256, N = 256, K = 8) issued by the
// leader (cluster rank 0). Each CTA loads only its own 128 rows of A and its
// half (128 rows) of B, hi and lo: 32 KB per stage instead of 48 KB, six
// stages. Synchronisation as in the bf16 2-SM kernel: the leader's full
// barrier counts both CTAs' bytes; MMA commits are multicast to both CTAs'
// empty and accumulator barriers; both CTAs' epilogue warps release an
// accumulator on the leader's tempty barrier (count 8). Each CTA's TMEM holds
// its 128 rows x 256 columns, so the epilogue is the 1-SM one.
constexpr int STAGES2 = 6;
constexpr uint32_t B2_BYTES = (BN / 2) * BK * 4;                 // 8 KB: this CTA's half of B
constexpr uint32_t STAGE2_BYTES = 2 * A_BYTES + 2 * B2_BYTES;    // 32 KB
constexpr uint32_t PAIR_STAGE2_BYTES = 2 * STAGE2_BYTES;
constexpr size_t SMEM2_BYTES = 1024 + size_t(STAGES2) * STAGE2_BYTES + 256;

// Work item t -> (bucket, matrix, this CTA's tile row tm, column tile tn):
// pairs of tile rows (2q, 2q + 1); symmetric phases visit column tiles tn >= q.
template <int PHASE, typename P>
__device__ __forceinline__ void decode_pair32(const P& p, long long t, uint32_t rank, int& b, int& mat, int& tm,
                                              int& tn) {
  b = 0;
  while (b + 1 < p.nb && t >= p.bk[b + 1].tile_begin) ++b;
  const Gemm32Bucket& B = p.bk[b];
  const long long local = t - B.tile_begin;
  mat = static_cast<int>(local / B.tiles_per_mat);
  int r = static_cast<int>(local % B.tiles_per_mat);
  int q;
  if (PHASE == PH32_BXT) {
    q = r / B.tiles_n;
    tn = r % B.tiles_n;
  } else {
    q = 0;
    while (true) {
      const int cnt = B.tiles_n - q;
      if (r < cnt) {
        tn = q + r;
        break;
      }
      r -= cnt;
      ++q;
    }
  }
  tm = 2 * q + static_cast<int>(rank);
}

template <int PHASE, bool FINAL, typename P>
__global__ void __launch_bounds__(THREADS, 1) ns_gemm32_pair_kernel(const __grid_constant__ P p) {
  static_assert(!FINAL || PHASE == PH32_BXT, "only the B*X phase has a final-store form");
  constexpr uint32_t IDESC = idesc_make(2u, 2 * BM, BN, false, false);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // stage s: [A hi | A lo | B hi half | B lo half]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES2 * STAGE2_BYTES);
  uint64_t* empty = full + STAGES2;
  uint64_t* tfull = empty + STAGES2;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  if (blockDim.x != THREADS) {
    if (threadIdx.x == 0) atomicOr(p.status, NS_DEV_BAD_LAUNCH);
    return;
  }
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const long long t0 = static_cast<long long>(cluster_id_x());
  const long long tstride = static_cast<long long>(cluster_count_x());

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES2; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 8);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    for (int b = 0; b < p.nb; ++b) {
      prefetch_tmap(&p.tmah[b]);
      prefetch_tmap(&p.tmal[b]);
      prefetch_tmap(&p.tmbh[b]);
      prefetch_tmap(&p.tmbl[b]);
    }
  }
  // the collective 2-SM TMEM allocation needs the peer CTA running: meet first
  __syncthreads();
  cluster_sync_all();
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers and TMEM exist before any cross-CTA traffic
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  griddep_wait();
  griddep_launch_dependents();

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer
    uint32_t stage = 0, phase = 0;
    long long issued = 0;
    for (long long t = t0; t < p.total_tiles; t += tstride) {
      int b, mat, tm, tn;
      decode_pair32<PHASE>(p, t, rank, b, mat, tm, tn);
      const int kb_n = p.bk[b].k_blocks;
      const int n0 = tn * BN + static_cast<int>(rank) * (BN / 2);
      for (int kb = 0; kb < kb_n; ++kb) {
        if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.status)) goto producer_done;
        const uint32_t full_l = map_to_rank(&full[stage], 0);
        if (leader) mbar_arrive_expect_tx(&full[stage], PAIR_STAGE2_BYTES);
        uint8_t* base = smem + stage * STAGE2_BYTES;
        tma_load_3d_pair(base, &p.tmah[b], full_l, kb * BK, tm * BM, mat);
        tma_load_3d_pair(base + A_BYTES, &p.tmal[b], full_l, kb * BK, tm * BM, mat);
        tma_load_3d_pair(base + 2 * A_BYTES, &p.tmbh[b], full_l, kb * BK, n0, mat);
        tma_load_3d_pair(base + 2 * A_BYTES + B2_BYTES, &p.tmbl[b], full_l, kb * BK, n0, mat);
        ++issued;
        if (++stage == STAGES2) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  producer_done:
    if (*abort_flag && leader) {
      const long long first = issued > STAGES2 ? issued - STAGES2 : 0;
      for (long long i = first; i < issued; ++i)
        mbar_wait_drain(&full[i % STAGES2], static_cast<uint32_t>((i / STAGES2) & 1), p.status);
    }
  } else if (warp == 1 && lane == 0 && leader) {
    // ----------------------------------------------------------- MMA issuer
    uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
    for (long long t = t0; t < p.total_tiles; t += tstride) {
      int b, mat, tm, tn;
      decode_pair32<PHASE>(p, t, rank, b, mat, tm, tn);
      const int kb_n = p.bk[b].k_blocks;
      if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag, p.status)) goto mma_done;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * BN;
      for (int kb = 0; kb < kb_n; ++kb) {
        if (!mbar_wait(&full[stage], phase, abort_flag, p.status)) goto mma_done;
        tc_fence_after();
        const uint32_t ah = smem_u32(smem + stage * STAGE2_BYTES);
        const uint32_t al = ah + A_BYTES;
        const uint32_t bh = ah + 2 * A_BYTES;
        const uint32_t bl = bh + B2_BYTES;
#pragma unroll
        for (int k = 0; k < BK / UK; ++k) {
          const uint32_t o = k * (UK * 4);  // 32 bytes per K step inside the 64-byte row
          const uint32_t first = (kb | k) != 0 ? 1u : 0u;
          mma_tf32_pair(d_tmem, sdesc_sw64(ah + o, 16, 512), sdesc_sw64(bh + o, 16, 512), IDESC, first);
          mma_tf32_pair(d_tmem, sdesc_sw64(ah + o, 16, 512), sdesc_sw64(bl + o, 16, 512), IDESC, 1u);
          mma_tf32_pair(d_tmem, sdesc_sw64(al + o, 16, 512), sdesc_sw64(bh + o, 16, 512), IDESC, 1u);
        }
        mma_commit_pair_mc(&empty[stage], 3);  // both CTAs' copies of the stage are free
        if (++stage == STAGES2) {
          stage = 0;
          phase ^= 1u;
        }
      }
      mma_commit_pair_mc(&tfull[acc], 3);
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
  mma_done:
    if (*abort_flag) {
      mma_commit_pair_mc(drain, 1);
      mbar_wait_drain(drain, 0, p.status);
    }
  } else if (warp >= 2) {
    // -------------------------------------------------------------- epilogue
    const int lg = warp & 3;
    uint32_t acc = 0, acc_phase = 0;
    const uint32_t tempty_leader0 = map_to_rank(&tempty[0], 0);
    const uint32_t tempty_leader1 = map_to_rank(&tempty[1], 0);
    for (long long t = t0; t < p.total_tiles; t += tstride) {
      int b, mat, tm, tn;
      decode_pair32<PHASE>(p, t, rank, b, mat, tm, tn);
      if (!mbar_wait(&tfull[acc], acc_phase, abort_flag, p.status)) break;
      tc_fence_after();
      epilogue32_tile<PHASE, FINAL>(p, b, mat, tm, tn, tmem_base, acc, lg, lane);
      tc_fence_before();
      __syncwarp();
      // the leader's MMA waits for all 8 epilogue warps of the pair
      if (lane == 0) mbar_arrive_cluster(acc ? tempty_leader1 : tempty_leader0);
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both CTAs done: no more multicast arrivals or remote arrives
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
  __syncthreads();
  cluster_sync_all();
}

template <int PHASE, bool FINAL, typename P>
cudaError_t launch32_pair(const P& p, int nsm, cudaStream_t st) {
  auto kern = ns_gemm32_pair_kernel<PHASE, FINAL, P>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(SMEM2_BYTES));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = SMEM2_BYTES;
  cfg.stream = st;
  cfg.gridDim = dim3(static_cast<unsigned>(2 * (nsm / 2)));
  int max_clusters = 0;
  e = cudaOccupancyMaxActiveClusters(&max_clusters, kern, &cfg);
  if (e != cudaSuccess) return e;
  if (max_clusters < 1) return cudaErrorInvalidConfiguration;
  const long long items = std::min<long long>(p.total_tiles, 1 << 30);
  cfg.gridDim = dim3(static_cast<unsigned>(2 * std::min<long long>(items, max_clusters)));
  e = cudaLaunchKernelEx(&cfg, kern, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int PHASE, bool FINAL, typename P>
cudaError_t launch32(const P& p, int grid, cudaStream_t st) {
  auto kern = ns_gemm32_kernel<PHASE, FINAL, P>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(SMEM_BYTES));
  if (e != cudaSuccess) return e;
  e = launch_pdl(kern, dim3(grid), dim3(THREADS), SMEM_BYTES, st, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// Trace ridge r = ridge * trace(A) / m, one CTA per matrix (fixed-order
// reduction). Standard step: A <- A + r I on the (hi, lo) pair. Gram-space
// step (coef set): write that matrix's Q coefficients instead.
__global__ void __launch_bounds__(256) ns_ridge32_kernel(const __grid_constant__ Ridge32Params p) {
  griddep_wait();
  griddep_launch_dependents();
  const Ridge32Bucket& B = p.bk[blockIdx.y];
  if (static_cast<int>(blockIdx.x) >= B.count) return;
  float* ah = B.ah + static_cast<long long>(blockIdx.x) * B.mat_stride;
  float* al = B.al + static_cast<long long>(blockIdx.x) * B.mat_stride;
  __shared__ double red[256];
  double s = 0.0;
  for (int i = threadIdx.x; i < B.m; i += blockDim.x) {
    const long long d = static_cast<long long>(i) * B.ld + i;
    s += static_cast<double>(ah[d]) + static_cast<double>(al[d]);
  }
  red[threadIdx.x] = s;
  __syncthreads();
  for (int o = blockDim.x / 2; o > 0; o >>= 1) {
    if (threadIdx.x < o) red[threadIdx.x] += red[threadIdx.x + o];
    __syncthreads();
  }
  const double rr = static_cast<double>(p.ridge) * red[0] / B.m;
  if (p.coef[blockIdx.y]) {
    // Gram-space step: Q = aI + b(A + rI) + c(A + rI)^2
    //                    = (a + b r + c r^2) I + (b + 2 c r) A + c A^2
    if (threadIdx.x == 0) {
      float* cf = p.coef[blockIdx.y] + 3 * blockIdx.x;
      cf[0] = static_cast<float>(p.a + p.b * rr + p.c * rr * rr);
      cf[1] = static_cast<float>(p.b + 2.0 * p.c * rr);
      cf[2] = p.c;
    }
    return;
  }
  const float delta = static_cast<float>(rr);
  __syncthreads();
  for (int i = threadIdx.x; i < B.m; i += blockDim.x) {
    const long long d = static_cast<long long>(i) * B.ld + i;
    const float v = ah[d] + al[d] + delta;
    const float h = tf32_round(v);
    ah[d] = h;
    al[d] = v - h;
  }
}

}  // namespace

cudaError_t launch_gemm32(int phase, const Gemm32Params& p, int nsm, cudaStream_t st) {
  if (p.total_tiles <= 0) return cudaSuccess;
  if (p.pair) {
    switch (phase) {
      case PH32_GRAM: return launch32_pair<PH32_GRAM, false>(p, nsm, st);
      case PH32_A2B: return launch32_pair<PH32_A2B, false>(p, nsm, st);
      case PH32_BXT: return launch32_pair<PH32_BXT, false>(p, nsm, st);
      default: return cudaErrorInvalidValue;
    }
  }
  const int grid = static_cast<int>(std::min<long long>(p.total_tiles, nsm));
  switch (phase) {
    case PH32_GRAM: return launch32<PH32_GRAM, false>(p, grid, st);
    case PH32_A2B: return launch32<PH32_A2B, false>(p, grid, st);
    case PH32_BXT: return launch32<PH32_BXT, false>(p, grid, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_gemm32_final(const Gemm32FinalParams& p, int nsm, cudaStream_t st) {
  if (p.total_tiles <= 0) return cudaSuccess;
  if (p.pair) return launch32_pair<PH32_BXT, true>(p, nsm, st);
  return launch32<PH32_BXT, true>(p, static_cast<int>(std::min<long long>(p.total_tiles, nsm)), st);
}

cudaError_t launch_ridge32(const Ridge32Params& p, cudaStream_t st) {
  if (p.nb <= 0 || p.max_count <= 0) return cudaSuccess;
  const cudaError_t e = launch_pdl(ns_ridge32_kernel, dim3(p.max_count, p.nb), dim3(256), 0, st, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace nsk
