// bf16 Newton-Schulz orchestration: GEMM launch parameters per phase (tensor
// maps, bucket tables, tiling choice, serpentine order), the one-pass
// prologue and the k steps with the final store. Megatron-Core API page
// owner_planning (ns_cost_fn) and Megatron-LM issue #6720 (shape-batched NS,
// SYRK-style symmetric products): tensors of equal (m, n) form a bucket laid
// out as one [count, m_pad, n_pad] array in the caller's workspace, and every
// phase of every step runs as one persistent launch over the tiles of all
// buckets of a group.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <mutex>
#include <vector>

#include "orchestrate.h"
#include "status.h"

namespace nsorch {

// Upper-triangle work items of one matrix: single tiles (cl = 1) or pairs of
// tile rows 2q, 2q + 1 sharing their column tiles (cl = 2, the 2-SM MMA).
long long syrk_tiles(int tiles_m, int tiles_n, int cl) {
  long long t = 0;
  if (cl == 1) {
    for (int tm = 0; tm < tiles_m; ++tm) t += tiles_n - (tm * nsk::GEMM_BM) / nsk::GEMM_BN;
  } else {
    for (int q = 0; q < (tiles_m + 1) / 2; ++q) t += tiles_n - q;
  }
  return t;
}

namespace {

// GEMM tiling for a launch: 1 = one CTA per 128 x 256 tile; 3 = CTA pairs
// running the 2-SM MMA on 256 x 256 tiles. Pairs need every bucket of the
// launch to have at least two tile rows.
int pick_cl(const Plan& p, size_t b0, size_t b1, int phase) {
  for (size_t bi = b0; bi < b1; ++bi) {
    const Bucket& b = p.buckets[bi];
    if (b.m_pad / nsk::GEMM_BM < 2) return 1;
  }
  if (const int f = gemm_cluster_override()) return f;
  // Measured (interleaved runs on one plan): the 2-SM MMA is faster for the
  // Gram (K = n) and A*A everywhere, and for B*X when every bucket has an even
  // number of tile rows (GPT-style and Llama-shaped: 16 and 32 rows); with an
  // odd count the spare half of the last pair makes the 1-SM kernel faster
  // for B*X (MoE 1408-row experts: 11 rows).
  if (phase == nsk::PH_BX)
    for (size_t bi = b0; bi < b1; ++bi)
      if ((p.buckets[bi].m_pad / nsk::GEMM_BM) % 2) return 1;
  return 3;
}

// Work items per matrix count tile-row pairs in the paired mode.
int count_mode(int cl) { return cl == 1 ? 1 : 2; }

}  // namespace

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

namespace {

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
        // both operands are A (upper pair blocks): rows through tma, the
        // transposed blocks left of the diagonal through tmt (A) and tmb (B)
        rc = make_map(&gp.tma[nb], q.a, b.m_pad, b.m_pad, cnt, 64, 128);
        if (rc == NS_OK) rc = make_map(&gp.tmt[nb], q.a, b.m_pad, b.m_pad, cnt, 64, 64);
        if (rc == NS_OK) rc = make_map(&gp.tmb[nb], q.a, b.m_pad, b.m_pad, cnt, 64, 64);
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
      if (rc == NS_OK) rc = make_map(&gp.tmt[nb], q.b, b.m_pad, b.m_pad, cnt, 64, 64);
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
              unsigned int* status, bool first_step, bool reverse, bool mirror, cudaStream_t st) {
  nsk::GemmParams gp;
  const int cl = pick_cl(p, b0, b1, phase);
  int rc = fill_phase(gp, p, ws, phase, cur_is_x0, b0, b1, status, nullptr, count_mode(cl), first_step);
  if (rc != NS_OK) return rc;
  gp.reverse = reverse ? 1 : 0;
  gp.mirror = mirror ? 1 : 0;
  if (const unsigned long long ns = take_gemm_stall()) {
    gp.stall = 1;
    gp.wait_ns = ns;
  }
  return counted(phase, st, [&] {
           return cl == 3 ? nsk::launch_gemm_pair(phase, gp, nsm, st) : nsk::launch_gemm(phase, gp, nsm, st);
         }) == cudaSuccess
             ? NS_OK
             : NS_ERR_CUDA;
}

// B*X phase of the last step, storing results directly into `out`, or with
// rank_out (row shards along dim 0) into the S rank buffers.
int run_final_bx(const Plan& p, char* ws, bool cur_is_x0, size_t b0, size_t b1, int nsm, unsigned int* status,
                 void* const* out, bool first_step, bool reverse, bool mirror, cudaStream_t st,
                 void* const* rank_out = nullptr) {
  static thread_local nsk::GemmFinalParams gp;  // ~32 KB: kept off the stack
  const int cl = pick_cl(p, b0, b1, nsk::PH_BX);
  int rc = fill_phase(gp, p, ws, nsk::PH_BX, cur_is_x0, b0, b1, status, out, count_mode(cl), first_step, rank_out);
  gp.reverse = reverse ? 1 : 0;
  gp.mirror = mirror ? 1 : 0;
  if (rc != NS_OK) return rc;
  if (const unsigned long long ns = take_gemm_stall()) {
    gp.stall = 1;
    gp.wait_ns = ns;
  }
  return counted(K_BX_FINAL, st, [&] {
           return cl == 3 ? nsk::launch_gemm_pair_final(gp, nsm, st) : nsk::launch_gemm_final(gp, nsm, st);
         }) == cudaSuccess
             ? NS_OK
             : NS_ERR_CUDA;
}

}  // namespace

size_t group_matrices(const Plan& p, size_t b0, size_t b1) {
  size_t n = 0;
  for (size_t bi = b0; bi < b1; ++bi) n += p.buckets[bi].members.size();
  return n;
}

// bf16 path, part 1: sums of squares, scales, X_0 = scale * (T or T^T),
// zero padded into the workspace.
// With rank_in (row-shard plans, shard_dim 0) the rows are read straight from
// the S rank buffers, which fuses the pack to the home buffers away; `in` is
// then unused.
int prologue_bf16(const Plan& p, const void* const* in, void* const* out, char* ws, unsigned int* status,
                  cudaStream_t st, const void* const* rank_in) {
  // prologue: X~_0 = T or T^T (unscaled, zero padded) with per-block sums of
  // squares in one pass, then the scales (GEMM buckets only: the small ones
  // load their inputs themselves)
  const size_t ng = gemm_buckets(p);
  for (size_t bi = 0; bi < ng; ++bi) {
    const Bucket& b = p.buckets[bi];
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

size_t gemm_buckets(const Plan& p) {
  if (!small_path_enabled()) return p.buckets.size();
  size_t n = 0;
  while (n < p.buckets.size() && !p.buckets[n].small) ++n;
  return n;
}

// Whether every bucket group's last B*X launch can store its results itself
// (its per-matrix table fits the parameter block) and there is a last step;
// small buckets always store their own results.
bool final_stores_all(const Plan& p) {
  const size_t ng = gemm_buckets(p);
  if (ng == 0) return true;
  if (p.steps == 0) return false;
  for (size_t b0 = 0; b0 < ng; b0 += nsk::GEMM_MAX_BUCKETS)
    if (group_matrices(p, b0, std::min(ng, b0 + nsk::GEMM_MAX_BUCKETS)) > size_t(nsk::GEMM_MAX_OUT))
      return false;
  return true;
}

int small_bf16(const Plan& p, const void* const* in, void* const* out, unsigned int* status, cudaStream_t st,
               const void* const* rank_in, void* const* rank_out) {
  const size_t ng = gemm_buckets(p);
  if (ng == p.buckets.size()) return NS_OK;
  static thread_local nsk::SmallParams sp;  // ~21 KB: kept off the stack
  auto launch = [&]() -> int {
    if (sp.count == 0) return NS_OK;
    const int rc = counted(K_SMALL, st, [&] { return nsk::launch_small(sp, st); }) == cudaSuccess ? NS_OK : NS_ERR_CUDA;
    sp.count = 0;
    sp.n_pad = 0;
    return rc;
  };
  std::memset(&sp, 0, sizeof(sp));
  sp.steps = p.steps;
  sp.a = p.a;
  sp.b = p.b;
  sp.c = p.c;
  sp.eps = p.eps;
  sp.status = status;
  sp.S = p.S;
  sp.in_ranks = rank_in ? 1 : 0;
  sp.out_ranks = rank_out ? 1 : 0;
  for (int r = 0; r < p.S && r < nsk::ROUTE_MAX_RANKS; ++r) {
    sp.rank_in[r] = rank_in ? rank_in[r] : nullptr;
    sp.rank_out[r] = rank_out ? rank_out[r] : nullptr;
  }
  for (size_t bi = ng; bi < p.buckets.size(); ++bi) {
    const Bucket& b = p.buckets[bi];
    for (int i : b.members) {
      const Tensor& t = p.t[i];
      if (sp.count == nsk::SMALL_MAX_MATS) {
        const int rc = launch();
        if (rc != NS_OK) return rc;
      }
      nsk::SmallMat& mt = sp.mat[sp.count++];
      mt.in = rank_in ? nullptr : in[t.ordinal];
      mt.out = rank_out ? nullptr : out[t.ordinal];
      mt.rank_off = t.rank_off;
      mt.rows = static_cast<int>(t.rows);
      mt.cols = static_cast<int>(t.cols);
      mt.transposed = t.transposed ? 1 : 0;
      sp.n_pad = std::max(sp.n_pad, static_cast<int>(b.n_pad));
    }
  }
  return launch();
}

// bf16 path, part 2: k steps of (Gram, A*A + B, B*X) and the final store.
// With rank_out (row shards along dim 0, final_stores_all(p)) the results go
// straight to the S rank buffers, fusing the unpack away; `out` is then unused.
int steps_bf16(const Plan& p, void* const* out, char* ws, int nsm, unsigned int* status, cudaStream_t st,
               void* const* rank_out) {
  if (rank_out && !final_stores_all(p)) return NS_ERR_ARG;
  int rc = NS_OK;
  // k steps x (Gram, A*A + B, B*X) over all buckets. The last B*X launch of
  // a bucket group writes the results straight to `out` when its per-matrix
  // table fits the parameter block; other groups go through the store kernel.
  const size_t ng = gemm_buckets(p);
  std::vector<char> stored(ng, 0);
  // one storage mode for every product of the call
  const bool mirror = symmetric_mirror();
  bool cur_is_x0 = true;
  for (int step = 0; step < p.steps; ++step) {
    const bool last = step + 1 == p.steps;
    for (int phase = nsk::PH_GRAM; phase <= nsk::PH_BX; ++phase) {
      for (size_t b0 = 0; b0 < ng; b0 += nsk::GEMM_MAX_BUCKETS) {
        const size_t b1 = std::min(ng, b0 + nsk::GEMM_MAX_BUCKETS);
        // serpentine order: every other product walks its tiles backwards,
        // starting on the matrices the previous product wrote last (still in L2)
        const bool serp = ((step * 3 + phase) & 1) != 0;
        if (last && phase == nsk::PH_BX && group_matrices(p, b0, b1) <= size_t(nsk::GEMM_MAX_OUT)) {
          rc = run_final_bx(p, ws, cur_is_x0, b0, b1, nsm, status, out, step == 0, serp, mirror, st, rank_out);
          for (size_t bi = b0; bi < b1; ++bi) stored[bi] = 1;
        } else {
          rc = run_phase(p, ws, phase, cur_is_x0, b0, b1, nsm, status, step == 0, serp, mirror, st);
        }
        if (rc != NS_OK) return rc;
      }
    }
    cur_is_x0 = !cur_is_x0;
  }
  // transpose back and store (buckets not stored by the last B*X launch)
  for (size_t bi = 0; bi < ng; ++bi) {
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

}  // namespace nsorch
