// Epilogue warps of the bf16 Newton-Schulz GEMM kernels (gemm.cu, gemm2sm.cu).
//
// Each of the four epilogue warps owns 32 TMEM lanes, i.e. 32 rows of the
// CTA's 128 x 256 fp32 accumulator, and walks them in 32 x 32 chunks. The
// epilogue of the three products (Megatron-Core API page owner_planning,
// ns_cost_fn; the quintic step of the layer_sharded_a2a page):
//
//   PH_GRAM  out = acc                      (A = X X^T)
//   PH_A2B   out = b * aux + c * acc        (B = b A + c A^2, aux = A)
//   PH_BX    out = a * aux + acc            (X' = a X + B X, aux = X)
//
// In the first step X is the unscaled X~_0 and the per-matrix scale
// s = 1 / (||T||_F + eps) enters here: out = s^2 acc (Gram) and
// out = s (a aux + acc) (B*X), i.e. the step run on X_0 = s X~_0.
//
// Data movement is staged through shared memory so that global memory only
// sees whole rows of a chunk:
//   * every warp has a ring of EPI_SLOTS chunk slots (32 rows x 64 bytes,
//     64-byte swizzle: 16-byte unit u of row y sits at u ^ ((y >> 1) & 3));
//   * lane 0 loads the aux chunk of job g + EPI_SLOTS - 1 by TMA while job g
//     is processed (jobs run on across tiles), completion on the slot's
//     mbarrier;
//   * lane i reads row i of the chunk from its slot (conflict-free with the
//     swizzle), combines it with TMEM columns of row i, writes the bf16 result
//     back to the same place, and lane 0 stores the slot by TMA;
//   * a slot is reloaded only after its store has finished reading it
//     (bulk-group wait), and generic accesses are fenced against the async
//     proxy before TMA touches the slot again.
// Symmetric phases store every chunk of the tiles they compute, which are
// exactly the upper 256 x 256 pair blocks of A or B (kernels.h). By default
// nothing is mirrored: the products that read A or B take the rest from the
// transposed blocks. With p.mirror, a tile right of its rows' diagonal pair
// block also writes its transpose straight to global memory (lanes hold
// consecutive rows: one contiguous 64-byte segment per store instruction);
// the diagonal pair blocks are computed in full and need no mirror.
// The final B*X launch writes each result to the caller's tensor (cropped,
// transposed back where needed) from registers instead of by TMA.
// Every wait is bounded; on a timeout or abort the warp stops, lets the loads
// it issued land and waits for its stores before returning.
#pragma once

#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace nsk {

using namespace nsptx;

constexpr int EPI_WARPS = 4;
constexpr int EPI_SLOTS = 4;
constexpr uint32_t EPI_SLOT_BYTES = 32 * 32 * 2;
constexpr uint32_t EPI_RING_BYTES = EPI_WARPS * EPI_SLOTS * EPI_SLOT_BYTES;  // 32 KB

struct EpiTile {
  int b, mat, tm, tn;
  int ci_hi;  // this warp's chunks [0, ci_hi) of the tile
};

// Tile t -> its chunks for the warp owning rows [tm*128 + 32*lg, +32).
template <int PHASE, typename P, typename Dec>
__device__ __forceinline__ EpiTile epi_tile(const P& p, const Dec& dec, long long t, int lg) {
  EpiTile e;
  dec(t, e.b, e.mat, e.tm, e.tn);
  const GemmBucket& B = p.bk[e.b];
  const int c_base = e.tn * GEMM_BN;
  // a pair's second row past the last tile row (odd tiles_m) stores nothing
  e.ci_hi = e.tm < B.tiles_m ? min(GEMM_BN / 32, (B.cols_valid - c_base) / 32) : 0;
  return e;
}

// Job cursor over (tile, chunk) in the order the warp consumes them.
struct EpiCursor {
  long long t;
  int ci;
  EpiTile e;
};

template <int PHASE, typename P, typename Dec>
__device__ __forceinline__ bool epi_next(const P& p, const Dec& dec, EpiCursor& c, long long tstride, int lg) {
  ++c.ci;
  while (c.ci >= c.e.ci_hi) {
    c.t += tstride;
    if (c.t >= p.total_tiles) return false;
    c.e = epi_tile<PHASE>(p, dec, c.t, lg);
    c.ci = 0;
  }
  return true;
}

__device__ __forceinline__ uint32_t epi_pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Byte offset of 16-byte unit u of row y in a 64-byte-swizzled slot.
__device__ __forceinline__ uint32_t epi_swz(int y, int u) {
  return static_cast<uint32_t>(y * 64 + ((u ^ ((y >> 1) & 3)) << 4));
}

// ring: this warp's EPI_SLOTS slots; rfull: their mbarriers (count 1).
// release(acc): signal that TMEM accumulator `acc` may be overwritten.
template <int PHASE, bool FINAL, typename P, typename Dec, typename Release>
__device__ __forceinline__ void epilogue_warp(const P& p, const Dec& dec, const Release& release, uint32_t tmem_base,
                                              int lg, int lane, long long t0, long long tstride, uint64_t lim,
                                              uint64_t* tfull,
                                              uint8_t* ring, uint64_t* rfull, volatile int* abort_flag) {
  constexpr bool SYRK = PHASE != PH_BX;
  constexpr bool AUX = PHASE != PH_GRAM;
  // loads run EPI_SLOTS - 1 jobs ahead of the job being processed
  EpiCursor ld;
  ld.t = t0 - tstride;
  ld.ci = 0;
  ld.e.ci_hi = 0;
  long long issued = 0, g = 0;
  bool more = AUX ? epi_next<PHASE>(p, dec, ld, tstride, lg) : false;
  auto issue = [&]() {
    const int s = static_cast<int>(issued % EPI_SLOTS);
    mbar_arrive_expect_tx(&rfull[s], EPI_SLOT_BYTES);
    tma_load_3d(ring + s * EPI_SLOT_BYTES, &p.tme[ld.e.b], &rfull[s], ld.e.tn * GEMM_BN + ld.ci * 32,
                ld.e.tm * GEMM_BM + lg * 32, ld.e.mat);
    ++issued;
    more = epi_next<PHASE>(p, dec, ld, tstride, lg);
  };
  if (AUX && lane == 0)
    while (more && issued < EPI_SLOTS - 1) issue();

  uint32_t acc = 0, acc_phase = 0;
  bool ok = true;
  for (long long t = t0; ok && t < p.total_tiles; t += tstride) {
    const EpiTile e = epi_tile<PHASE>(p, dec, t, lg);
    const GemmBucket& B = p.bk[e.b];
    // waits are warp-uniform: a lane that timed out stops the whole warp
    const bool got = mbar_wait(&tfull[acc], acc_phase, abort_flag, p.status, lim);
    if (!__all_sync(0xffffffffu, got)) {
      ok = false;
      break;
    }
    tc_fence_after();
    if (e.ci_hi == 0) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) release(acc);
    }
    const int r0w = e.tm * GEMM_BM + lg * 32;
    const int r = r0w + lane;
    // first step: X~_0 is unscaled, s = 1 / (||T||_F + eps) per matrix
    const float sc = (PHASE != PH_A2B && B.scale) ? B.scale[e.mat] : 1.0f;
    for (int ci = 0; ci < e.ci_hi; ++ci, ++g) {
      const int s = static_cast<int>(g % EPI_SLOTS);
      uint8_t* slot = ring + s * EPI_SLOT_BYTES;
      const int cg = e.tn * GEMM_BN + ci * 32;
      if (AUX) {
        const bool got = mbar_wait(&rfull[s], static_cast<uint32_t>((g / EPI_SLOTS) & 1), abort_flag, p.status, lim);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
      } else {
        // the slot's previous store (job g - EPI_SLOTS) has read it
        if (lane == 0) bulk_wait_group_read<EPI_SLOTS - 1>();
        __syncwarp();
      }
      uint32_t v[32];
      tmem_ld32(tmem_base + (static_cast<uint32_t>(lg * 32) << 16) + acc * GEMM_BN + ci * 32, v);
      tmem_ld_wait();
      if (ci + 1 == e.ci_hi) {
        // the accumulator is in registers: the MMA may start the next tile
        tc_fence_before();
        __syncwarp();
        if (lane == 0) release(acc);
      }
      float f[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) f[j] = __uint_as_float(v[j]);
      if (PHASE == PH_GRAM) {
        const float sc2 = sc * sc;
#pragma unroll
        for (int j = 0; j < 32; ++j) f[j] *= sc2;
      }
      if (AUX) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint4 q = *reinterpret_cast<const uint4*>(slot + epi_swz(lane, u));
          const uint32_t w4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float x0 = __uint_as_float(w4[k] << 16), x1 = __uint_as_float(w4[k] & 0xFFFF0000u);
            float& f0 = f[u * 8 + 2 * k];
            float& f1 = f[u * 8 + 2 * k + 1];
            if (PHASE == PH_A2B) {
              f0 = p.beta * x0 + p.gamma * f0;
              f1 = p.beta * x1 + p.gamma * f1;
            } else {
              f0 = sc * (p.alpha * x0 + f0);
              f1 = sc * (p.alpha * x1 + f1);
            }
          }
        }
      }
      uint32_t w[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) w[j] = epi_pack_bf16(f[2 * j], f[2 * j + 1]);
      const __nv_bfloat16* hv = reinterpret_cast<const __nv_bfloat16*>(w);
      if (FINAL) {
        // row r of X_k (m index), columns cg.. (n index) -> the caller's tensor
        if (r < B.m_valid) {
          const unsigned long long en = p.out_tab[B.out_first + e.mat];
          if (!p.out_ranks) {
            __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(en & ~1ull);
            if (!(en & 1ull)) {
              __nv_bfloat16* dst = o + static_cast<long long>(r) * B.n_valid + cg;
              if (cg + 32 <= B.n_valid && (reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
                uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
                for (int u = 0; u < 4; ++u) d4[u] = make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
              } else {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                  if (cg + j < B.n_valid) dst[j] = hv[j];
              }
            } else {
              // transposed tensor: element (r, c) of X_k is element (c, r) of
              // the output; lanes hold consecutive r, so each store is contiguous
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (cg + j < B.n_valid) o[static_cast<long long>(cg + j) * B.m_valid + r] = hv[j];
            }
          } else {
            // row shards along dim 0: row j of the output tensor is row
            // j % sh of the shard at offset en >> 1 of rank buffer j / sh
            const long long off = static_cast<long long>(en >> 1);
            if (!(en & 1ull)) {
              const int sh = B.m_valid / p.S;
              const int rk = r / sh;
              __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(p.rank_ptr[rk]) + off +
                                   static_cast<long long>(r - rk * sh) * B.n_valid + cg;
              if (cg + 32 <= B.n_valid && (reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
                uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
                for (int u = 0; u < 4; ++u) d4[u] = make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
              } else {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                  if (cg + j < B.n_valid) dst[j] = hv[j];
              }
            } else {
              // transposed: output rows cg .. cg + 31
              const int sh = B.n_valid / p.S;
              int rk = cg / sh, lr = cg - rk * sh;
              if (lr + 32 <= sh) {
                // all 32 rows in one shard (always when sh is a multiple of
                // 32): one base pointer, contiguous stores as for a tensor
                __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(p.rank_ptr[rk]) + off +
                                   static_cast<long long>(lr) * B.m_valid + r;
#pragma unroll
                for (int j = 0; j < 32; ++j)
                  if (cg + j < B.n_valid) o[static_cast<long long>(j) * B.m_valid] = hv[j];
              } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                  if (cg + j < B.n_valid)
                    reinterpret_cast<__nv_bfloat16*>(p.rank_ptr[rk])[off + static_cast<long long>(lr) * B.m_valid + r] =
                        hv[j];
                  if (++lr == sh) {
                    ++rk;
                    lr = 0;
                  }
                }
              }
            }
          }
        }
        // every lane's slot reads are done before the slot is reloaded
        fence_proxy_async_smem();
        __syncwarp();
      } else {
#pragma unroll
        for (int u = 0; u < 4; ++u)
          *reinterpret_cast<uint4*>(slot + epi_swz(lane, u)) = make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_3d(&p.tmo[e.b], slot, cg, r0w, e.mat);
          bulk_commit_group();
        }
        if (SYRK && p.mirror && e.tn > e.tm / 2) {
          // right of the diagonal pair block: (r, c) also goes to (c, r)
          __nv_bfloat16* o =
              reinterpret_cast<__nv_bfloat16*>(B.out) + static_cast<long long>(e.mat) * B.out_stride;
#pragma unroll
          for (int j = 0; j < 32; ++j) o[static_cast<long long>(cg + j) * B.ld_out + r] = hv[j];
        }
      }
      if (AUX && lane == 0 && more) {
        // the next load reuses the slot of job g - 1, whose store was
        // committed before this job's
        bulk_wait_group_read<1>();
        issue();
      }
    }
    acc ^= 1u;
    if (acc == 0) acc_phase ^= 1u;
  }
  if (lane == 0) {
    // loads issued but not consumed (abort only) land before the CTA exits
    for (long long i = g; i < issued; ++i)
      mbar_wait_drain(&rfull[i % EPI_SLOTS], static_cast<uint32_t>((i / EPI_SLOTS) & 1), p.status);
    bulk_wait_group<0>();
  }
  __syncwarp();
}

}  // namespace nsk
