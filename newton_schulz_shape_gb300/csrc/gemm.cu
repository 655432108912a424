// The three tensor-core products of one quintic Newton-Schulz step
// (Megatron-Core API page owner_planning, ns_cost_fn):
//
//   PH_GRAM  A = X X^T                  symmetric: upper pair blocks only
//   PH_A2B   B = b A + c (A A)          symmetric: upper pair blocks only
//   PH_BX    X' = a X + B X             full tiles, written to the other X buffer
//
// A and B are stored as their upper 256 x 256 pair blocks (kernels.h). A·A
// and B·X read their symmetric operands K-block by K-block: left of the
// operand rows' diagonal pair block from the transposed, stored block
// (MN-major loads, transposed MMA operand), elsewhere as rows (K-major).
// The TMA producer and the MMA issuer therefore walk a tile's K-blocks in at
// most three runs (both operands transposed, A as rows, both as rows), each
// with its layout fixed at compile time: both are single threads that the
// tensor pipe waits on, and choosing the layout per K-block at run time slowed
// them measurably.
//
// One persistent kernel per phase, one CTA per SM, a 128 x 256 output tile per
// work item, tiles of every shape bucket of the launch in one static schedule,
// walked first to last or (p.reverse) last to first: successive launches
// alternate, so each starts on the matrices its predecessor wrote last, which
// are still in L2.
// Warp roles (192 threads):
//   warp 0 lane 0   TMA producer: K-blocks of 64 into a 4-stage smem ring
//   warp 1          TMEM allocator; lane 0 issues tcgen05.mma (M=128, N=256,
//                   K=16, bf16 in, fp32 accumulate) and commits to mbarriers
//   warps 2-5       epilogue (epilogue.cuh): tcgen05.ld of the accumulator (two
//                   TMEM buffers of 256 columns, so the next tile's MMAs
//                   overlap), fused scalar epilogue in fp32, chunks staged in
//                   shared memory and moved by TMA
// Operands: X, A, B are zero-padded in the workspace (rows to 128, cols to
// 64), so every K-block is full and the MMA needs no masking; tiles that hang
// over the padded edge read TMA's zero fill and skip their stores.
#include <cuda_bf16.h>

#include <algorithm>
#include <type_traits>

#include "epilogue.cuh"
#include "kernels.h"
#include "launch.cuh"
#include "ptx.cuh"

namespace nsk {
namespace {

using namespace nsptx;

constexpr int BM = GEMM_BM, BN = GEMM_BN, BK = GEMM_BK, UK = 16;
constexpr int STAGES = 4;
constexpr uint32_t A_BYTES = BM * BK * 2;  // 16 KB
constexpr uint32_t B_BYTES = BN * BK * 2;  // 32 KB
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
constexpr uint32_t TMEM_COLS = 2 * BN;  // two fp32 accumulators of 128 lanes x 256 columns
constexpr int THREADS = 192;
constexpr size_t SMEM_BYTES = 1024 + size_t(STAGES) * STAGE_BYTES + EPI_RING_BYTES + 512;

// Work item t -> (bucket b, matrix, output tile (tm, tn)). SYRK phases visit
// only tiles that touch the upper triangle: in tile row tm, column tiles from
// floor(tm * BM / BN).
template <int PHASE, typename P>
__device__ __forceinline__ void decode_tile(const P& p, long long t, int& b, int& mat, int& tm, int& tn) {
  if (p.reverse) t = p.total_tiles - 1 - t;
  b = 0;
  while (b + 1 < p.nb && t >= p.bk[b + 1].tile_begin) ++b;
  const GemmBucket& B = p.bk[b];
  const long long local = t - B.tile_begin;
  mat = static_cast<int>(local / B.tiles_per_mat);
  int r = static_cast<int>(local % B.tiles_per_mat);
  if (PHASE == PH_BX) {
    tm = r / B.tiles_n;
    tn = r % B.tiles_n;
    return;
  }
  tm = 0;
  while (true) {
    const int tn0 = (tm * BM) / BN;
    const int cnt = B.tiles_n - tn0;
    if (r < cnt) {
      tn = tn0 + r;
      return;
    }
    r -= cnt;
    ++tm;
  }
}

// FINAL (B*X phase only): write the cropped, transposed-back result to the
// caller's tensors listed in p.out_tab instead of the next X buffer.
template <int PHASE, bool FINAL, typename P>
__global__ void __launch_bounds__(THREADS, 1) ns_gemm_kernel(const __grid_constant__ P p) {
  static_assert(!FINAL || PHASE == PH_BX, "only the B*X phase has a final-store form");
  // symmetric operands stored as upper pair blocks: A of A*A and B*X, B of A*A
  constexpr bool A_TRI = (PHASE != PH_GRAM);
  constexpr bool B_TRI = (PHASE == PH_A2B);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_BYTES;
  uint8_t* ring = smem + STAGES * STAGE_BYTES;  // epilogue chunk slots
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + EPI_RING_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint64_t* rfull = drain + 1;  // EPI_WARPS x EPI_SLOTS
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(rfull + EPI_WARPS * EPI_SLOTS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  if (blockDim.x != THREADS) {
    if (threadIdx.x == 0) atomicOr(p.status, NS_DEV_BAD_LAUNCH);
    return;
  }
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const long long t0 = static_cast<long long>(blockIdx.x);
  const long long tstride = static_cast<long long>(gridDim.x);

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
    for (int i = 0; i < EPI_WARPS * EPI_SLOTS; ++i) mbar_init(&rfull[i], 1);
    *abort_flag = 0;
    fence_mbar_init();
    for (int b = 0; b < p.nb; ++b) {
      prefetch_tmap(&p.tma[b]);
      prefetch_tmap(&p.tmb[b]);
      if (PHASE != PH_GRAM) {
        prefetch_tmap(&p.tme[b]);
        prefetch_tmap(&p.tmt[b]);
      }
      if (!FINAL) prefetch_tmap(&p.tmo[b]);
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
  const uint64_t lim = p.wait_ns ? p.wait_ns : NS_WAIT_LIMIT_NS;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer
    uint32_t stage = 0, phase = 0;
    long long issued = 0;
    for (long long t = p.stall ? p.total_tiles : t0; t < p.total_tiles; t += tstride) {
      int b, mat, tm, tn;
      decode_tile<PHASE>(p, t, b, mat, tm, tn);
      const int kb_n = p.bk[b].k_blocks;
      // K-blocks left of the operand rows' diagonal pair block come transposed
      const int kb_ta = A_TRI && !p.mirror ? (tm / 2) * (2 * BM / BK) : 0;
      const int kb_tb = B_TRI && !p.mirror ? tn * (BN / BK) : 0;
      // K-blocks [kb0, kb1) with one operand layout, fixed at compile time:
      // layout choices made per K-block at run time slowed this single thread
      // enough to leave the ring short of operands
      auto load = [&](auto a_mn_c, auto b_mn_c, int kb0, int kb1) -> bool {
        constexpr bool AMN = decltype(a_mn_c)::value, BMN = decltype(b_mn_c)::value;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.status, lim)) return false;
          mbar_arrive_expect_tx(&full[stage], STAGE_BYTES);
          uint8_t* a_dst = sA + stage * A_BYTES;
          uint8_t* b_dst = sB + stage * B_BYTES;
          if (AMN) {
#pragma unroll
            for (int j = 0; j < BM / 64; ++j)
              tma_load_3d(a_dst + j * (64 * 128), &p.tmt[b], &full[stage], tm * BM + j * 64, kb * BK, mat);
          } else {
            tma_load_3d(a_dst, &p.tma[b], &full[stage], kb * BK, tm * BM, mat);
          }
          if (!BMN) {
            // K-major rows: X (Gram), or A through the A operand's map (A*A)
            const CUtensorMap* mb = PHASE == PH_GRAM ? &p.tmb[b] : &p.tma[b];
            tma_load_3d(b_dst, mb, &full[stage], kb * BK, tn * BN, mat);
            tma_load_3d(b_dst + 128 * 128, mb, &full[stage], kb * BK, tn * BN + 128, mat);
          } else {
#pragma unroll
            for (int j = 0; j < BN / 64; ++j)
              tma_load_3d(b_dst + j * (64 * 128), &p.tmb[b], &full[stage], tn * BN + j * 64, kb * BK, mat);
          }
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        return true;
      };
      using T_ = std::true_type;
      using F_ = std::false_type;
      bool ok;
      if (PHASE == PH_BX)
        ok = load(T_{}, T_{}, 0, kb_ta) && load(F_{}, T_{}, kb_ta, kb_n);
      else if (PHASE == PH_GRAM)
        ok = load(F_{}, F_{}, 0, kb_n);
      else
        ok = load(T_{}, T_{}, 0, kb_ta) && load(F_{}, T_{}, kb_ta, kb_tb) && load(F_{}, F_{}, kb_tb, kb_n);
      if (!ok) goto producer_done;
    }
  producer_done:
    if (*abort_flag) {
      // let the copies already issued land before the CTA exits
      const long long first = issued > STAGES ? issued - STAGES : 0;
      for (long long i = first; i < issued; ++i)
        mbar_wait_drain(&full[i % STAGES], static_cast<uint32_t>((i / STAGES) & 1), p.status);
    }
  } else if (warp == 1 && lane == 0) {
    // ----------------------------------------------------------- MMA issuer
    uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
    for (long long t = t0; t < p.total_tiles; t += tstride) {
      int b, mat, tm, tn;
      decode_tile<PHASE>(p, t, b, mat, tm, tn);
      const int kb_n = p.bk[b].k_blocks;
      if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag, p.status, lim)) goto mma_done;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * BN;
      const int kb_ta = A_TRI && !p.mirror ? (tm / 2) * (2 * BM / BK) : 0;
      const int kb_tb = B_TRI && !p.mirror ? tn * (BN / BK) : 0;
      // K-blocks [kb0, kb1) with one operand layout, fixed at compile time
      auto run = [&](auto a_mn_c, auto b_mn_c, int kb0, int kb1) -> bool {
        constexpr bool AMN = decltype(a_mn_c)::value, BMN = decltype(b_mn_c)::value;
        constexpr uint32_t IDESC = idesc_make(1u, BM, BN, AMN, BMN);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag, p.status, lim)) return false;
          tc_fence_after();
          const uint32_t a_addr = smem_u32(sA + stage * A_BYTES);
          const uint32_t b_addr = smem_u32(sB + stage * B_BYTES);
#pragma unroll
          for (int k = 0; k < BK / UK; ++k) {
            const uint64_t ad = AMN ? sdesc_sw128(a_addr + k * (UK * 128), 64 * 128, 1024)
                                    : sdesc_sw128(a_addr + k * (UK * 2), 16, 1024);
            const uint64_t bd = BMN ? sdesc_sw128(b_addr + k * (UK * 128), 64 * 128, 1024)
                                    : sdesc_sw128(b_addr + k * (UK * 2), 16, 1024);
            mma_f16(d_tmem, ad, bd, IDESC, (kb | k) != 0 ? 1u : 0u);
          }
          mma_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        return true;
      };
      using T_ = std::true_type;
      using F_ = std::false_type;
      // at most three runs: both operands transposed, then A as rows, then both as rows
      bool ok;
      if (PHASE == PH_BX)
        ok = run(T_{}, T_{}, 0, kb_ta) && run(F_{}, T_{}, kb_ta, kb_n);
      else if (PHASE == PH_GRAM)
        ok = run(F_{}, F_{}, 0, kb_n);
      else
        ok = run(T_{}, T_{}, 0, kb_ta) && run(F_{}, T_{}, kb_ta, kb_tb) && run(F_{}, F_{}, kb_tb, kb_n);
      if (!ok) goto mma_done;
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
    const int lg = warp & 3;  // this warp may read TMEM lanes [32*lg, 32*lg + 32)
    auto dec = [&](long long t, int& b, int& mat, int& tm, int& tn) {
      decode_tile<PHASE>(p, t, b, mat, tm, tn);
    };
    auto release = [&](uint32_t a) { mbar_arrive(&tempty[a]); };
    epilogue_warp<PHASE, FINAL>(p, dec, release, tmem_base, lg, lane, t0, tstride, lim, tfull,
                                ring + lg * EPI_SLOTS * EPI_SLOT_BYTES, rfull + lg * EPI_SLOTS, abort_flag);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

template <int PHASE, bool FINAL, typename P>
cudaError_t launch_one(const P& p, int work_items, int nsm, cudaStream_t st) {
  auto kern = ns_gemm_kernel<PHASE, FINAL, P>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(SMEM_BYTES));
  if (e != cudaSuccess) return e;
  e = launch_pdl(kern, dim3(static_cast<unsigned>(std::min(work_items, nsm))), dim3(THREADS), SMEM_BYTES, st, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm(int phase, const GemmParams& p, int nsm, cudaStream_t st) {
  if (p.total_tiles <= 0) return cudaSuccess;
  const int items = static_cast<int>(std::min<long long>(p.total_tiles, 1 << 30));
  switch (phase) {
    case PH_GRAM: return launch_one<PH_GRAM, false>(p, items, nsm, st);
    case PH_A2B: return launch_one<PH_A2B, false>(p, items, nsm, st);
    case PH_BX: return launch_one<PH_BX, false>(p, items, nsm, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_gemm_final(const GemmFinalParams& p, int nsm, cudaStream_t st) {
  if (p.total_tiles <= 0) return cudaSuccess;
  const int items = static_cast<int>(std::min<long long>(p.total_tiles, 1 << 30));
  return launch_one<PH_BX, true>(p, items, nsm, st);
}

}  // namespace nsk
