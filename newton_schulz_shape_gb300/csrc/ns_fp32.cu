// fp32-Gram Newton-Schulz orchestration (NS_FP32_GRAM): split-TF32 (hi, lo)
// operands, the trace ridge, and its Gram-space form (NS_FP32_GRAM_SPACE,
// Megatron-LM issue #6720 gram_once). NS_FP32_AUTO runs both on views of one
// plan (api.cu).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <mutex>
#include <vector>

#include "orchestrate.h"
#include "status.h"

namespace nsorch {
namespace {

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

// 3-D fp32 tensor map over [count][outer][inner], box {GEMM32_BK, 128, 1}, 64-byte swizzle.
int make_map32(CUtensorMap* m, void* base, uint64_t inner, uint64_t outer, uint64_t count) {
  cuuint64_t dims[3] = {inner, outer, count};
  cuuint64_t strides[2] = {inner * 4, inner * outer * 4};
  cuuint32_t box[3] = {nsk::GEMM32_BK, 128, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = tensor_map_encoder()(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? NS_OK : NS_ERR_CUDA;
}

// The 2-SM form (pairs of 128-row tiles on a cluster of two CTAs) for a
// launch whose buckets all have at least two tile rows in the phase's M
// dimension (m_pad for the symmetric products, n_pad for (B X)^T), unless the
// 1-SM tiling is forced (ns_set_gemm_cluster(1)). Both give identical bits.
bool pair32(const Plan& p, size_t b0, size_t b1, int phase) {
  if (gemm_cluster_override() == 1) return false;
  for (size_t bi = b0; bi < b1; ++bi) {
    const Bucket& b = p.buckets[bi];
    const int64_t rows = phase == nsk::PH32_BXT ? b.n_pad : b.m_pad;
    if (rows / nsk::GEMM_BM < 2) return false;
  }
  return true;
}

template <typename P>
int fill_phase32(P& gp, const Plan& p, char* ws, int phase, int cur, size_t b0, size_t b1, unsigned int* status,
                 void* const* final_out) {
  std::memset(&gp, 0, sizeof(gp));
  gp.alpha = p.a;
  gp.beta = p.b;
  gp.gamma = p.c;
  gp.status = status;
  gp.pair = pair32(p, b0, b1, phase) ? 1 : 0;
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
      g.tiles_per_mat = static_cast<int>(syrk_tiles(g.tiles_m, g.tiles_n, gp.pair ? 2 : 1));
      g.ld = static_cast<int>(b.m_pad);
      g.mat_stride = b.m_pad * b.m_pad;
      if (phase == nsk::PH32_GRAM) {
        float* xh = q.x[cur];
        float* xl = xh + q.xs;
        g.k_blocks = static_cast<int>(b.n_pad / nsk::GEMM32_BK);
        g.out_h = q.a;
        g.out_l = q.a + q.as;
        rc = make_map32(&gp.tmah[nb], xh, b.n_pad, b.m_pad, cnt);
        if (rc == NS_OK) rc = make_map32(&gp.tmal[nb], xl, b.n_pad, b.m_pad, cnt);
        if (rc == NS_OK) rc = make_map32(&gp.tmbh[nb], xh, b.n_pad, b.m_pad, cnt);
        if (rc == NS_OK) rc = make_map32(&gp.tmbl[nb], xl, b.n_pad, b.m_pad, cnt);
      } else {
        g.k_blocks = static_cast<int>(b.m_pad / nsk::GEMM32_BK);
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
      g.tiles_per_mat = (gp.pair ? (g.tiles_m + 1) / 2 : g.tiles_m) * g.tiles_n;
      g.k_blocks = static_cast<int>(b.m_pad / nsk::GEMM32_BK);
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
  gp.pair = pair32(p, b0, b1, nsk::PH32_A2B) ? 1 : 0;
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
    g.tiles_per_mat = static_cast<int>(syrk_tiles(g.tiles_m, g.tiles_n, gp.pair ? 2 : 1));
    g.ld = static_cast<int>(b.m_pad);
    g.mat_stride = b.m_pad * b.m_pad;
    g.k_blocks = static_cast<int>(b.m_pad / nsk::GEMM32_BK);
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
  return counted(nsk::PH32_A2B, st, [&] { return nsk::launch_gemm32(nsk::PH32_A2B, gp, nsm, st); }) ==
                 cudaSuccess
             ? NS_OK
             : NS_ERR_CUDA;
}


}  // namespace

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
      if (counted(nsk::PH32_GRAM, st, [&] { return nsk::launch_gemm32(nsk::PH32_GRAM, gp, nsm, st); }) !=
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
      if (counted(K_BX_FINAL, st, [&] { return nsk::launch_gemm32_final(gp, nsm, st); }) != cudaSuccess)
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
          if (counted(K_BX_FINAL, st, [&] { return nsk::launch_gemm32_final(gp, nsm, st); }) != cudaSuccess)
            return NS_ERR_CUDA;
          for (size_t bi = b0; bi < b1; ++bi) stored[bi] = 1;
        } else {
          nsk::Gemm32Params gp;
          rc = fill_phase32(gp, p, ws, phase, cur, b0, b1, status, nullptr);
          if (rc != NS_OK) return rc;
          if (counted(phase, st, [&] { return nsk::launch_gemm32(phase, gp, nsm, st); }) != cudaSuccess)
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

}  // namespace nsorch
