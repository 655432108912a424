// 2-SM (cta_group::2) form of the three bf16 Newton-Schulz products (see
// gemm.cu for the phases and their epilogues; Megatron-Core API page
// owner_planning, ns_cost_fn).
//
// A cluster of two CTAs computes one 256 x 256 output tile with
// tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 16) issued by one thread of
// the leader CTA (cluster rank 0). Each CTA holds, per 64-wide K block, only
// its own half of each operand: A rows [tm*128, +128) with tm = 2q + rank, and
// B rows (or columns) [tn*256 + rank*128, +128): 32 KB per stage per SM,
// against 48 KB when one SM holds a whole 128 x 256 tile's operands. The
// accumulator is split by rows: each CTA's TMEM holds its 128 rows x 256
// fp32 columns, so each CTA's epilogue works exactly as in the 1-SM kernel.
// A and B are stored as upper pair blocks (kernels.h): the K-blocks of a
// symmetric operand left of its rows' diagonal pair block are loaded MN-major
// from the transposed block, and the MMA takes that operand transposed. Both
// CTAs' A rows lie in pair row q and their B rows in pair row tn, so the
// choice is the same in both halves of every MMA.
// In a diagonal pair tile of A*A (tn == q) each CTA's B rows are its own A
// rows, in the same layout: only A is loaded and the MMA reads B from the A
// stage. (The Gram's diagonal tiles could do the same, but the Gram does not
// wait for its operands, and reading both from one stage made its MMAs a
// little slower.)
//
// Synchronisation (all waits bounded):
//   full[s]   leader only; count 1 (the leader's arrive.expect_tx of both
//             halves' bytes); both CTAs' TMA loads signal it with complete_tx.
//             The peer's bytes for a phase can only be issued after the
//             leader's MMA released the previous phase, so they never land in
//             the wrong phase; the peer needs no arrive (and no fence).
//   empty[s]  both CTAs; the leader's MMA commit is multicast to both
//   tfull[a]  both CTAs; the leader's commit after a tile, multicast
//   tempty[a] leader only; count 8 = 4 epilogue warps x 2 CTAs (remote arrive)
// TMEM is allocated and freed collectively by one warp in each CTA.
#include <cuda_bf16.h>

#include <algorithm>
#include <type_traits>

#include "epilogue.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace nsk {
namespace {

using namespace nsptx;

constexpr int BM = GEMM_BM;          // rows per CTA (M = 256 per pair)
constexpr int BN = GEMM_BN;          // output columns per tile
constexpr int BK = GEMM_BK, UK = 16;
constexpr int STAGES = 6;
constexpr uint32_t A_BYTES = BM * BK * 2;         // 16 KB: this CTA's 128 rows of A
constexpr uint32_t B_BYTES = (BN / 2) * BK * 2;   // 16 KB: this CTA's half of B
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
constexpr uint32_t PAIR_STAGE_BYTES = 2 * STAGE_BYTES;
constexpr uint32_t TMEM_COLS = 2 * BN;
constexpr int THREADS = 192;
constexpr size_t SMEM_BYTES = 1024 + size_t(STAGES) * STAGE_BYTES + EPI_RING_BYTES + 512;

template <int PHASE, typename P>
__device__ __forceinline__ void decode_pair(const P& p, long long t, uint32_t rank, int& b, int& mat, int& tm,
                                            int& tn) {
  if (p.reverse) t = p.total_tiles - 1 - t;
  b = 0;
  while (b + 1 < p.nb && t >= p.bk[b + 1].tile_begin) ++b;
  const GemmBucket& B = p.bk[b];
  const long long local = t - B.tile_begin;
  mat = static_cast<int>(local / B.tiles_per_mat);
  int r = static_cast<int>(local % B.tiles_per_mat);
  int q;
  if (PHASE == PH_BX) {
    q = r / B.tiles_n;
    tn = r % B.tiles_n;
  } else {
    // 256-row block q touches the upper triangle in column tiles tn >= q
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
__global__ void __launch_bounds__(THREADS, 1) ns_gemm2sm_kernel(const __grid_constant__ P p) {
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
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const long long t0 = static_cast<long long>(cluster_id_x());
  const long long tstride = static_cast<long long>(cluster_count_x());

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 8);
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
      decode_pair<PHASE>(p, t, rank, b, mat, tm, tn);
      const int kb_n = p.bk[b].k_blocks;
      // K-blocks left of the operand rows' diagonal pair block come transposed
      const int kb_ta = A_TRI && !p.mirror ? (tm / 2) * (2 * BM / BK) : 0;
      const int kb_tb = B_TRI && !p.mirror ? tn * (BN / BK) : 0;
      const bool diag = PHASE == PH_A2B && tn == tm / 2;  // B rows == A rows
      // K-blocks [kb0, kb1) with one operand layout (and, for DG, no B load),
      // fixed at compile time: layout choices made per K-block at run time
      // slowed this single thread enough to leave the ring short of operands
      auto load = [&](auto a_mn_c, auto b_mn_c, auto dg_c, int kb0, int kb1) -> bool {
        constexpr bool AMN = decltype(a_mn_c)::value, BMN = decltype(b_mn_c)::value, DG = decltype(dg_c)::value;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.status, lim)) return false;
          const uint32_t full_l = map_to_rank(&full[stage], 0);
          if (leader) mbar_arrive_expect_tx(&full[stage], DG ? 2 * A_BYTES : PAIR_STAGE_BYTES);
          uint8_t* a_dst = sA + stage * A_BYTES;
          if (AMN) {
#pragma unroll
            for (int j = 0; j < BM / 64; ++j)
              tma_load_3d_pair(a_dst + j * (64 * 128), &p.tmt[b], full_l, tm * BM + j * 64, kb * BK, mat);
          } else {
            tma_load_3d_pair(a_dst, &p.tma[b], full_l, kb * BK, tm * BM, mat);
          }
          // DG: the A stage holds this CTA's B rows already
          if (!DG) {
            uint8_t* b_dst = sB + stage * B_BYTES;
            const int n0 = tn * BN + static_cast<int>(rank) * (BN / 2);
            if (BMN) {
#pragma unroll
              for (int j = 0; j < BN / 128; ++j)
                tma_load_3d_pair(b_dst + j * (64 * 128), &p.tmb[b], full_l, n0 + j * 64, kb * BK, mat);
            } else {
              // K-major rows: X (Gram), or A through the A operand's map (A*A)
              tma_load_3d_pair(b_dst, PHASE == PH_GRAM ? &p.tmb[b] : &p.tma[b], full_l, kb * BK, n0, mat);
            }
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
        ok = load(T_{}, T_{}, F_{}, 0, kb_ta) && load(F_{}, T_{}, F_{}, kb_ta, kb_n);
      else if (PHASE == PH_GRAM)
        ok = load(F_{}, F_{}, F_{}, 0, kb_n);
      else if (diag)  // kb_ta == kb_tb here
        ok = load(T_{}, T_{}, T_{}, 0, kb_ta) && load(F_{}, F_{}, T_{}, kb_ta, kb_n);
      else
        ok = load(T_{}, T_{}, F_{}, 0, kb_ta) && load(F_{}, T_{}, F_{}, kb_ta, kb_tb) &&
             load(F_{}, F_{}, F_{}, kb_tb, kb_n);
      if (!ok) goto producer_done;
    }
  producer_done:
    if (*abort_flag && leader) {
      const long long first = issued > STAGES ? issued - STAGES : 0;
      for (long long i = first; i < issued; ++i)
        mbar_wait_drain(&full[i % STAGES], static_cast<uint32_t>((i / STAGES) & 1), p.status);
    }
  } else if (warp == 1 && lane == 0 && leader) {
    // ----------------------------------------------------------- MMA issuer
    uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
    for (long long t = t0; t < p.total_tiles; t += tstride) {
      int b, mat, tm, tn;
      decode_pair<PHASE>(p, t, rank, b, mat, tm, tn);
      const int kb_n = p.bk[b].k_blocks;
      if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag, p.status, lim)) goto mma_done;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * BN;
      const int kb_ta = A_TRI && !p.mirror ? (tm / 2) * (2 * BM / BK) : 0;
      const int kb_tb = B_TRI && !p.mirror ? tn * (BN / BK) : 0;
      const bool diag = PHASE == PH_A2B && tn == tm / 2;
      // K-blocks [kb0, kb1) with one operand layout, fixed at compile time so
      // that the issuing thread spends no instructions choosing descriptors
      auto run = [&](auto a_mn_c, auto b_mn_c, auto dg_c, int kb0, int kb1) -> bool {
        constexpr bool AMN = decltype(a_mn_c)::value, BMN = decltype(b_mn_c)::value, DG = decltype(dg_c)::value;
        constexpr uint32_t IDESC = idesc_make(1u, 2 * BM, BN, AMN, BMN);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag, p.status, lim)) return false;
          tc_fence_after();
          const uint32_t a_addr = smem_u32(sA + stage * A_BYTES);
          const uint32_t b_addr = DG ? a_addr : smem_u32(sB + stage * B_BYTES);
#pragma unroll
          for (int k = 0; k < BK / UK; ++k) {
            const uint64_t ad = AMN ? sdesc_sw128(a_addr + k * (UK * 128), 64 * 128, 1024)
                                    : sdesc_sw128(a_addr + k * (UK * 2), 16, 1024);
            const uint64_t bd = BMN ? sdesc_sw128(b_addr + k * (UK * 128), 64 * 128, 1024)
                                    : sdesc_sw128(b_addr + k * (UK * 2), 16, 1024);
            mma_f16_pair(d_tmem, ad, bd, IDESC, (kb | k) != 0 ? 1u : 0u);
          }
          mma_commit_pair_mc(&empty[stage], 3);  // both CTAs' copies of the stage are free
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
        ok = run(T_{}, T_{}, F_{}, 0, kb_ta) && run(F_{}, T_{}, F_{}, kb_ta, kb_n);
      else if (PHASE == PH_GRAM)
        ok = run(F_{}, F_{}, F_{}, 0, kb_n);
      else if (diag)  // kb_ta == kb_tb here
        ok = run(T_{}, T_{}, T_{}, 0, kb_ta) && run(F_{}, F_{}, T_{}, kb_ta, kb_n);
      else
        ok = run(T_{}, T_{}, F_{}, 0, kb_ta) && run(F_{}, T_{}, F_{}, kb_ta, kb_tb) &&
             run(F_{}, F_{}, F_{}, kb_tb, kb_n);
      if (!ok) goto mma_done;
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
    auto dec = [&](long long t, int& b, int& mat, int& tm, int& tn) {
      decode_pair<PHASE>(p, t, rank, b, mat, tm, tn);
    };
    // the leader's MMA waits for all 8 epilogue warps of the pair
    auto release = [&](uint32_t a) { mbar_arrive_cluster(map_to_rank(&tempty[a], 0)); };
    epilogue_warp<PHASE, FINAL>(p, dec, release, tmem_base, lg, lane, t0, tstride, lim, tfull,
                                ring + lg * EPI_SLOTS * EPI_SLOT_BYTES, rfull + lg * EPI_SLOTS, abort_flag);
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
cudaError_t launch_pair(const P& p, int work_items, int nsm, cudaStream_t st) {
  auto kern = ns_gemm2sm_kernel<PHASE, FINAL, P>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(SMEM_BYTES));
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
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = st;
  cfg.gridDim = dim3(static_cast<unsigned>(2 * (nsm / 2)));
  int max_clusters = 0;
  e = cudaOccupancyMaxActiveClusters(&max_clusters, kern, &cfg);
  if (e != cudaSuccess) return e;
  if (max_clusters < 1) return cudaErrorInvalidConfiguration;
  cfg.gridDim = dim3(static_cast<unsigned>(2 * std::min(work_items, max_clusters)));
  e = cudaLaunchKernelEx(&cfg, kern, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_pair(int phase, const GemmParams& p, int nsm, cudaStream_t st) {
  if (p.total_tiles <= 0) return cudaSuccess;
  const int items = static_cast<int>(std::min<long long>(p.total_tiles, 1 << 30));
  switch (phase) {
    case PH_GRAM: return launch_pair<PH_GRAM, false>(p, items, nsm, st);
    case PH_A2B: return launch_pair<PH_A2B, false>(p, items, nsm, st);
    case PH_BX: return launch_pair<PH_BX, false>(p, items, nsm, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_gemm_pair_final(const GemmFinalParams& p, int nsm, cudaStream_t st) {
  if (p.total_tiles <= 0) return cudaSuccess;
  const int items = static_cast<int>(std::min<long long>(p.total_tiles, 1 << 30));
  return launch_pair<PH_BX, true>(p, items, nsm, st);
}

}  // namespace nsk
