// Host planner: 2-D views, NS cost, greedy LPT homes/owners, routing offsets,
// shape buckets and the workspace layout. Pure host C++, no CUDA calls.
//
// Sources: Megatron-Core API pages core.distributed.fsdp.src.megatron_fsdp.
// experimental.owner_planning (ns_cost_fn, assign_owner_work, OwnerGatherPlan,
// OwnerScatterPlan) and core.optimizer.layer_sharded_a2a (params_by_home,
// route_to_ns_home, route_from_ns_home).
#include <algorithm>
#include <cstring>
#include <map>
#include <new>
#include <utility>

#include "../../include/nsgb300.h"
#include "plan.h"

namespace nsplan {

namespace {

bool mul_ok(int64_t a, int64_t b, int64_t* out) { return !__builtin_mul_overflow(a, b, out); }
bool add_ok(int64_t a, int64_t b, int64_t* out) { return !__builtin_add_overflow(a, b, out); }

int64_t round_up(int64_t v, int64_t q) { return (v + q - 1) / q * q; }

// owner_planning, ns_cost_fn: view (shape[0], prod(shape[1:])), cost
// numel * (min(rows, cols) * steps + 1).
int cost_of(const int64_t* shape, int ndim, int steps, int64_t* rows, int64_t* cols, int64_t* cost) {
  if (ndim < 2) return NS_ERR_SHAPE;
  for (int d = 0; d < ndim; ++d)
    if (shape[d] < 0) return NS_ERR_SHAPE;
  int64_t c = 1;
  for (int d = 1; d < ndim; ++d)
    if (!mul_ok(c, shape[d], &c)) return NS_ERR_ARG;
  int64_t numel, k, cst;
  if (!mul_ok(shape[0], c, &numel)) return NS_ERR_ARG;
  const int64_t mn = std::min(shape[0], c);
  if (!mul_ok(mn, steps, &k) || !add_ok(k, 1, &k) || !mul_ok(numel, k, &cst)) return NS_ERR_ARG;
  *rows = shape[0];
  *cols = c;
  *cost = cst;
  return NS_OK;
}

int load_tensors(Plan& p, int n, const int32_t* ndims, const int64_t* shapes, bool allow_1d) {
  p.t.assign(n, Tensor());
  int64_t pos = 0;
  for (int i = 0; i < n; ++i) {
    Tensor& t = p.t[i];
    const int nd = ndims[i];
    if (nd < 1 || nd > kMaxDims || (nd < 2 && !allow_1d)) return NS_ERR_SHAPE;
    t.ndim = nd;
    int64_t numel = 1;
    for (int d = 0; d < nd; ++d) {
      t.shape[d] = shapes[pos + d];
      if (t.shape[d] < 0) return NS_ERR_SHAPE;
      if (!mul_ok(numel, t.shape[d], &numel)) return NS_ERR_ARG;
    }
    t.numel = numel;
    if (nd >= 2) {
      int rc = cost_of(t.shape, nd, p.steps, &t.rows, &t.cols, &t.cost);
      if (rc != NS_OK) return rc;
      t.m = std::min(t.rows, t.cols);
      t.n = std::max(t.rows, t.cols);
      t.transposed = t.rows > t.cols;
    }
    pos += nd;
  }
  return NS_OK;
}

// Home buffers, buckets, workspace layout and routing table. keep_homes: a
// sub-plan of a pipeline wave keeps the whole plan's home offsets and sizes.
int finish(Plan& p, bool keep_homes = false) {
  // participating list and home offsets (increasing index order per home)
  p.part.clear();
  if (!keep_homes) p.home_sizes.assign(p.S, 0);
  for (size_t i = 0; i < p.t.size(); ++i) {
    Tensor& t = p.t[i];
    t.bucket = t.slot = -1;
    if (!t.participating) continue;
    t.ordinal = static_cast<int>(p.part.size());
    p.part.push_back(static_cast<int>(i));
    if (!keep_homes) {
      t.home_off = p.home_sizes[t.home];
      p.home_sizes[t.home] += t.numel;
    }
  }
  p.buckets.clear();
  // buckets of equal (m, n), heaviest per-matrix work first
  std::map<std::pair<int64_t, int64_t>, int> index;
  for (int i : p.part) {
    Tensor& t = p.t[i];
    if (t.numel == 0) continue;
    auto key = std::make_pair(t.m, t.n);
    auto it = index.find(key);
    if (it == index.end()) {
      Bucket b;
      b.m = t.m;
      b.n = t.n;
      b.m_pad = round_up(t.m, nsk::GEMM_BM);
      // fp32-Gram: n is also the M dimension of the (B X)^T product, tiled by 128
      b.n_pad = round_up(t.n, p.gram_mode != NS_BF16 ? nsk::GEMM_BM : nsk::GEMM_BK);
      index[key] = static_cast<int>(p.buckets.size());
      p.buckets.push_back(b);
      it = index.find(key);
    }
    p.buckets[it->second].members.push_back(i);
  }
  for (Bucket& b : p.buckets)
    b.small = p.gram_mode == NS_BF16 && b.m <= nsk::SMALL_MAX_M && b.n <= nsk::SMALL_MAX_N;
  std::stable_sort(p.buckets.begin(), p.buckets.end(), [](const Bucket& x, const Bucket& y) {
    // buckets that can run one CTA per matrix last (the GEMM launches then
    // cover a prefix), otherwise heaviest per-matrix work (~ m^2 n) first
    if (x.small != y.small) return y.small;
    const double wx = double(x.m) * double(x.m) * double(x.n);
    const double wy = double(y.m) * double(y.m) * double(y.n);
    return wx > wy;
  });
  // bf16 path: one bf16 copy of X per ping-pong buffer, A and B in bf16.
  // fp32-Gram path: X as (hi, lo) fp32 pairs, both m-major and transposed
  // (4 buffers per ping-pong set); A and B as (hi, lo) fp32 pairs.
  // fp32 Gram-space path: one X set, then (hi, lo) pairs of T, P0, P1 in the
  // second X region.
  const bool f32 = p.gram_mode != NS_BF16;
  const bool gs_all = p.gram_mode == NS_FP32_GRAM_SPACE;
  const bool gs_auto = p.gram_mode == NS_FP32_AUTO;
  const uint64_t xset = f32 ? 4 * 4 : 2;
  const uint64_t aset = f32 ? 2 * 4 : 2;
  uint64_t off = 0;
  auto take = [&](uint64_t bytes) {
    off = (off + 1023) / 1024 * 1024;
    uint64_t o = off;
    off += bytes;
    return o;
  };
  for (size_t bi = 0; bi < p.buckets.size(); ++bi) {
    Bucket& b = p.buckets[bi];
    const uint64_t cnt = b.members.size();
    for (size_t s = 0; s < b.members.size(); ++s) {
      p.t[b.members[s]].bucket = static_cast<int>(bi);
      p.t[b.members[s]].slot = static_cast<int>(s);
    }
    b.gram_space = gs_all || (gs_auto && b.n >= 2 * b.m);
    const bool gs = b.gram_space;
    const uint64_t xbytes = cnt * uint64_t(b.m_pad) * uint64_t(b.n_pad) * xset;
    const uint64_t abytes = cnt * uint64_t(b.m_pad) * uint64_t(b.m_pad) * aset;
    b.off_x0 = take(xbytes);
    b.off_x1 = take(gs ? cnt * uint64_t(b.m_pad) * uint64_t(b.m_pad) * 3 * aset : xbytes);
    b.off_a = take(abytes);
    b.off_b = take(abytes);
    // partial sums of squares per matrix: 32K-element chunks (fp32 paths) or
    // blocks of 64 rows x 1024 columns of the padded X_0 (bf16 path)
    b.nchunks = f32 ? (b.m * b.n + kSumsqChunk - 1) / kSumsqChunk : (b.m_pad / 64) * ((b.n_pad + 1023) / 1024);
    b.off_partial = take(cnt * uint64_t(b.nchunks) * 4);
    b.off_scale = take(cnt * 4);
    b.off_coef = take(cnt * 3 * 4);
  }
  p.ws_bytes = p.buckets.empty() ? 0 : (off + 1023) / 1024 * 1024;
  // routing table: one entry per participating tensor with data on the ranks
  p.route.clear();
  for (int i : p.part) {
    const Tensor& t = p.t[i];
    nsk::RouteEntry e{};
    e.home = t.home;
    e.home_off = t.home_off;
    if (p.layout != NS_LAYOUT_FLAT) {
      if (t.shard_len == 0) continue;
      e.seg_begin = t.rank_off;
      e.seg_len = t.shard_len;
      e.inner = t.run;
      e.outer = t.stride;
      e.mr = t.mr;
      e.mt = t.mt;
    } else {
      if (t.numel == 0) continue;
      e.seg_begin = t.flat_off;
      e.seg_len = t.numel;
      e.inner = 0;
      e.outer = 0;
    }
    p.route.push_back(e);
  }
  p.in_bytes = 2;
  p.out_bytes = p.gram_mode != NS_BF16 ? 4 : 2;
  return NS_OK;
}

}  // namespace

// NS-only sub-plan over `members` (tensor indices, increasing) of `base`:
// same tensors, homes and home offsets; buckets and workspace of the members.
int build_subplan(const Plan& base, const std::vector<int>& members, Plan& out) {
  out = base;
  for (Tensor& t : out.t) t.participating = false;
  for (int i : members) out.t[i].participating = true;
  for (void*& d : out.d_route) d = nullptr;  // device tables stay with the base plan
  int rc = finish(out, true);
  out.route.clear();
  return rc;
}

int lpt_assign(int n, const int64_t* costs, const int32_t* cand_ptr, const int32_t* cand_idx, int n_ranks,
               int32_t* owner_out) {
  if (n < 0 || n_ranks < 1 || (n > 0 && (!costs || !cand_ptr || !cand_idx || !owner_out))) return NS_ERR_ARG;
  if (n > 0 && cand_ptr[0] != 0) return NS_ERR_ARG;
  for (int i = 0; i < n; ++i) {
    if (costs[i] <= 0) return NS_ERR_ARG;
    if (cand_ptr[i + 1] < cand_ptr[i]) return NS_ERR_ARG;
    if (cand_ptr[i + 1] == cand_ptr[i]) return NS_ERR_HOME;
    for (int k = cand_ptr[i]; k < cand_ptr[i + 1]; ++k)
      if (cand_idx[k] < 0 || cand_idx[k] >= n_ranks) return NS_ERR_HOME;
  }
  // single-candidate tensors first (index order), then descending cost with
  // equal costs kept in index order (stable sort)
  std::vector<int> order;
  order.reserve(n);
  for (int i = 0; i < n; ++i)
    if (cand_ptr[i + 1] - cand_ptr[i] == 1) order.push_back(i);
  std::vector<int> multi;
  for (int i = 0; i < n; ++i)
    if (cand_ptr[i + 1] - cand_ptr[i] > 1) multi.push_back(i);
  std::stable_sort(multi.begin(), multi.end(), [&](int x, int y) { return costs[x] > costs[y]; });
  order.insert(order.end(), multi.begin(), multi.end());
  std::vector<int64_t> load(n_ranks, 0);
  for (int i : order) {
    int best = cand_idx[cand_ptr[i]];
    for (int k = cand_ptr[i] + 1; k < cand_ptr[i + 1]; ++k)
      if (load[cand_idx[k]] < load[best]) best = cand_idx[k];
    owner_out[i] = best;
    load[best] += costs[i];
  }
  return NS_OK;
}

int assign_homes_all(Plan& p, int n, int S, const int32_t* home_of);

int build_row_shard(Plan& p, int n, const int32_t* ndims, const int64_t* shapes, int S, int shard_dim,
                    const int32_t* home_of) {
  p.layout = NS_LAYOUT_ROW_SHARD;
  p.S = S;
  p.shard_dim = shard_dim;
  int rc = load_tensors(p, n, ndims, shapes, false);
  if (rc != NS_OK) return rc;
  int64_t pos = 0;
  for (int i = 0; i < n; ++i) {
    Tensor& t = p.t[i];
    if (shard_dim < 0 || shard_dim >= t.ndim) return NS_ERR_ARG;
    t.pre = 1;
    for (int d = 0; d < shard_dim; ++d) t.pre *= t.shape[d];
    t.D = t.shape[shard_dim];
    t.post = 1;
    for (int d = shard_dim + 1; d < t.ndim; ++d) t.post *= t.shape[d];
    if (t.D % S) return NS_ERR_NOT_DIVISIBLE;
    t.shard_len = t.numel / S;
    t.rank_off = pos;
    pos += t.shard_len;
    t.run = (t.D / S) * t.post;
    t.stride = t.D * t.post;
    t.mr = t.run;
    t.mt = 0;
    t.participating = true;
  }
  p.rank_len = pos;
  return assign_homes_all(p, n, S, home_of);
}

// Homes for the sharded models: explicit, or LPT with every rank a candidate
// (every rank holds a piece of every param).
int assign_homes_all(Plan& p, int n, int S, const int32_t* home_of) {
  int rc;
  if (home_of) {
    for (int i = 0; i < n; ++i) {
      if (home_of[i] < 0 || home_of[i] >= S) return NS_ERR_HOME;
      p.t[i].home = home_of[i];
    }
  } else if (n > 0) {
    // layer_sharded_a2a: every rank holds a shard of every param, so every
    // rank is a candidate home; owner_planning's LPT picks one.
    std::vector<int64_t> costs(n);
    std::vector<int32_t> ptr(n + 1), idx(int64_t(n) * S), own(n);
    for (int i = 0; i < n; ++i) {
      costs[i] = std::max<int64_t>(p.t[i].cost, 1);
      ptr[i] = i * S;
      for (int r = 0; r < S; ++r) idx[int64_t(i) * S + r] = r;
    }
    ptr[n] = n * S;
    rc = lpt_assign(n, costs.data(), ptr.data(), idx.data(), S, own.data());
    if (rc != NS_OK) return rc;
    for (int i = 0; i < n; ++i) p.t[i].home = own[i];
  }
  return finish(p);
}

int build_two_stage(Plan& p, int n, const int32_t* ndims, const int64_t* shapes, const int32_t* pdims, int R,
                    int T, const int32_t* home_of) {
  p.layout = NS_LAYOUT_TWO_STAGE;
  p.R = R;
  p.T = T;
  p.S = R * T;
  p.shard_dim = 0;
  int rc = load_tensors(p, n, ndims, shapes, false);
  if (rc != NS_OK) return rc;
  int64_t pos = 0;
  for (int i = 0; i < n; ++i) {
    Tensor& t = p.t[i];
    const int d = pdims[i];
    if (d < 0 || d >= t.ndim) return NS_ERR_ARG;
    const int64_t P = t.shape[0];
    int64_t pre = 1;  // dims strictly between 0 and d
    for (int k = 1; k < d; ++k) pre *= t.shape[k];
    const int64_t D = t.shape[d];
    int64_t post = 1;
    for (int k = d + 1; k < t.ndim; ++k) post *= t.shape[k];
    t.shard_len = t.numel / (int64_t(R) * T);
    if (d == 0) {
      // both stages split dim 0: TP slice t of P/T rows, remat slice r of it;
      // the piece of rank (r, t) is one contiguous block of rows
      if (P % (int64_t(R) * T)) return NS_ERR_NOT_DIVISIBLE;
      t.run = t.shard_len;
      t.stride = t.shard_len;
      t.mr = t.shard_len;
      t.mt = int64_t(R) * t.shard_len;
    } else {
      // TP slice t: columns [t*D/T, (t+1)*D/T) of dim d; remat slice r: rows
      // [r*P/R, (r+1)*P/R). Runs of (D/T)*post elements, one per (row, pre).
      if (P % R || D % T) return NS_ERR_NOT_DIVISIBLE;
      const int64_t cols = t.numel / std::max<int64_t>(P, 1);  // prod(shape[1:])
      t.run = (D / T) * post;
      t.stride = D * post;
      t.mr = (P / R) * cols;
      t.mt = (D / T) * post;
      (void)pre;
    }
    t.rank_off = pos;
    pos += t.shard_len;
    t.participating = true;
  }
  p.rank_len = pos;
  return assign_homes_all(p, n, p.S, home_of);
}

namespace {
bool piece(const Plan& p, int i, int r, int64_t* lo, int64_t* hi) {
  const int64_t per = p.buffer_size / p.S;
  const Tensor& t = p.t[i];
  *lo = std::max(t.flat_off, int64_t(r) * per);
  *hi = std::min(t.flat_off + t.numel, int64_t(r + 1) * per);
  return *lo < *hi;
}
}  // namespace

int build_flat(Plan& p, int n, const int32_t* ndims, const int64_t* shapes, const int64_t* offsets,
               int64_t size, const uint8_t* participating, int S, const int32_t* owner_of) {
  p.layout = NS_LAYOUT_FLAT;
  p.S = S;
  p.shard_dim = 0;
  if (size < 0) return NS_ERR_ARG;
  if (size % S) return NS_ERR_NOT_DIVISIBLE;
  p.buffer_size = size;
  p.rank_len = size / S;
  int rc = load_tensors(p, n, ndims, shapes, true);
  if (rc != NS_OK) return rc;
  int64_t prev_end = 0;
  for (int i = 0; i < n; ++i) {
    Tensor& t = p.t[i];
    t.flat_off = offsets[i];
    const bool part = participating ? participating[i] != 0 : t.ndim >= 2;
    if (!part) continue;
    if (t.ndim < 2 || t.numel == 0) return NS_ERR_SHAPE;
    if (t.flat_off < 0 || t.flat_off + t.numel > size) return NS_ERR_ARG;
    if (t.flat_off < prev_end) return NS_ERR_ARG;  // participating tensors in buffer order, disjoint
    prev_end = t.flat_off + t.numel;
    t.participating = true;
  }
  std::vector<int> part;
  for (int i = 0; i < n; ++i)
    if (p.t[i].participating) part.push_back(i);
  if (owner_of) {
    for (int i : part) {
      int64_t lo, hi;
      const int o = owner_of[i];
      if (o < 0 || o >= S || !piece(p, i, o, &lo, &hi)) return NS_ERR_HOME;
      p.t[i].home = o;
    }
  } else if (!part.empty()) {
    const int np = static_cast<int>(part.size());
    std::vector<int64_t> costs(np);
    std::vector<int32_t> ptr(np + 1, 0), idx, own(np);
    for (int k = 0; k < np; ++k) {
      costs[k] = std::max<int64_t>(p.t[part[k]].cost, 1);
      for (int r = 0; r < S; ++r) {
        int64_t lo, hi;
        if (piece(p, part[k], r, &lo, &hi)) idx.push_back(r);
      }
      ptr[k + 1] = static_cast<int32_t>(idx.size());
    }
    rc = lpt_assign(np, costs.data(), ptr.data(), idx.data(), S, own.data());
    if (rc != NS_OK) return rc;
    for (int k = 0; k < np; ++k) p.t[part[k]].home = own[k];
  }
  return finish(p);
}

int gather_meta(const Plan& p, int rho, int64_t* send, int64_t* recv, int64_t* roff, int64_t* own) {
  const int S = p.S;
  const int n = static_cast<int>(p.t.size());
  if (send)
    for (int r = 0; r < S; ++r) send[r] = 0;
  if (recv)
    for (int r = 0; r < S; ++r) recv[r] = 0;
  if (roff)
    for (int64_t k = 0; k < int64_t(n) * S; ++k) roff[k] = -1;
  if (own)
    for (int i = 0; i < n; ++i) own[i] = -1;
  for (int i = 0; i < n; ++i) {
    const Tensor& t = p.t[i];
    if (!t.participating) continue;
    int64_t lo, hi;
    if (t.home != rho) {
      if (piece(p, i, rho, &lo, &hi) && send) send[t.home] += hi - lo;
      continue;
    }
    if (own) own[i] = piece(p, i, rho, &lo, &hi) ? hi - lo : 0;
    for (int s = 0; s < S; ++s) {
      if (s == rho || !piece(p, i, s, &lo, &hi)) continue;
      // tensors owned by rho are laid out in index order in s's buffer to rho
      int64_t before = 0;
      for (int j = 0; j < i; ++j) {
        int64_t l2, h2;
        if (p.t[j].participating && p.t[j].home == rho && piece(p, j, s, &l2, &h2)) before += h2 - l2;
      }
      if (roff) roff[int64_t(i) * S + s] = before;
      if (recv) recv[s] += hi - lo;
    }
  }
  return NS_OK;
}

int scatter_meta(const Plan& p, int rho, int64_t* send, int64_t* recv, int64_t* roff) {
  const int S = p.S;
  const int n = static_cast<int>(p.t.size());
  if (send)
    for (int r = 0; r < S; ++r) send[r] = 0;
  if (recv)
    for (int r = 0; r < S; ++r) recv[r] = 0;
  if (roff)
    for (int64_t k = 0; k < int64_t(n) * S; ++k) roff[k] = -1;
  std::vector<int64_t> pos(S, 0);  // running offset inside each owner's buffer to rho
  for (int i = 0; i < n; ++i) {
    const Tensor& t = p.t[i];
    if (!t.participating) continue;
    int64_t lo, hi;
    if (t.home == rho) {
      for (int d = 0; d < S; ++d)
        if (d != rho && piece(p, i, d, &lo, &hi) && send) send[d] += hi - lo;
    } else if (piece(p, i, rho, &lo, &hi)) {
      if (roff) roff[int64_t(i) * S + t.home] = pos[t.home];
      pos[t.home] += hi - lo;
      if (recv) recv[t.home] += hi - lo;
    }
  }
  return NS_OK;
}

}  // namespace nsplan

using nsplan::Plan;

namespace {
int check_coeffs(int steps, float eps, int gram_mode, float ridge) {
  if (steps < 0) return NS_ERR_ARG;
  if (!(eps >= 0.0f)) return NS_ERR_ARG;
  if (gram_mode != NS_BF16 && gram_mode != NS_FP32_GRAM && gram_mode != NS_FP32_GRAM_SPACE &&
      gram_mode != NS_FP32_AUTO)
    return NS_ERR_ARG;
  if (!(ridge >= 0.0f)) return NS_ERR_ARG;
  if (gram_mode == NS_BF16 && ridge != 0.0f) return NS_ERR_ARG;
  return NS_OK;
}
// NS_FP32_AUTO: split the plan's buckets into the standard-fp32 and the
// Gram-space view. Each view keeps every tensor (ordinals index the caller's
// pointer arrays) and the buckets' workspace offsets.
void make_mode_views(ns_plan* pl) {
  if (pl->p.gram_mode != NS_FP32_AUTO) return;
  pl->view_std = pl->p;
  pl->view_gs = pl->p;
  pl->view_std.buckets.clear();
  pl->view_gs.buckets.clear();
  for (const nsplan::Bucket& b : pl->p.buckets) (b.gram_space ? pl->view_gs : pl->view_std).buckets.push_back(b);
  for (nsplan::Plan* v : {&pl->view_std, &pl->view_gs}) {
    v->route.clear();  // views never route
    for (int d = 0; d < nsplan::kMaxDevices; ++d) v->d_route[d] = nullptr;
  }
}
}  // namespace

extern "C" {

int ns_cost(const int64_t* shape, int ndim, int steps, int64_t* cost_out) {
  if (!shape || !cost_out || steps < 0) return NS_ERR_ARG;
  int64_t r, c;
  return nsplan::cost_of(shape, ndim, steps, &r, &c, cost_out);
}

int ns_assign_owner_work(int n_tensors, const int64_t* costs, const int32_t* cand_ptr, const int32_t* cand_idx,
                         int n_ranks, int32_t* owner_out) {
  return nsplan::lpt_assign(n_tensors, costs, cand_ptr, cand_idx, n_ranks, owner_out);
}

int ns_plan_create(int n_tensors, const int32_t* ndims, const int64_t* shapes_flat, int steps, float a, float b,
                   float c, float eps, int gram_mode, float ridge, int S, int shard_dim, const int32_t* home_of,
                   ns_plan_t** plan_out) {
  if (!plan_out) return NS_ERR_ARG;
  *plan_out = nullptr;
  if (n_tensors < 0 || (n_tensors > 0 && (!ndims || !shapes_flat))) return NS_ERR_ARG;
  if (S < 1 || S > nsplan::kMaxRanks) return NS_ERR_ARG;
  int rc = check_coeffs(steps, eps, gram_mode, ridge);
  if (rc != NS_OK) return rc;
  ns_plan* pl = new (std::nothrow) ns_plan();
  if (!pl) return NS_ERR_ARG;
  Plan& p = pl->p;
  p.steps = steps;
  p.a = a;
  p.b = b;
  p.c = c;
  p.eps = eps;
  p.gram_mode = gram_mode;
  p.ridge = ridge;
  rc = nsplan::build_row_shard(p, n_tensors, ndims, shapes_flat, S, shard_dim, home_of);
  if (rc != NS_OK) {
    delete pl;
    return rc;
  }
  make_mode_views(pl);
  *plan_out = pl;
  return NS_OK;
}

int ns_plan_create_two_stage(int n_tensors, const int32_t* ndims, const int64_t* shapes_flat,
                             const int32_t* partition_dims, int R, int T, int steps, float a, float b, float c,
                             float eps, int gram_mode, float ridge, const int32_t* home_of, ns_plan_t** plan_out) {
  if (!plan_out) return NS_ERR_ARG;
  *plan_out = nullptr;
  if (n_tensors < 0 || (n_tensors > 0 && (!ndims || !shapes_flat || !partition_dims))) return NS_ERR_ARG;
  if (R < 1 || T < 1 || int64_t(R) * T > nsplan::kMaxRanks) return NS_ERR_ARG;
  int rc = check_coeffs(steps, eps, gram_mode, ridge);
  if (rc != NS_OK) return rc;
  ns_plan* pl = new (std::nothrow) ns_plan();
  if (!pl) return NS_ERR_ARG;
  Plan& p = pl->p;
  p.steps = steps;
  p.a = a;
  p.b = b;
  p.c = c;
  p.eps = eps;
  p.gram_mode = gram_mode;
  p.ridge = ridge;
  rc = nsplan::build_two_stage(p, n_tensors, ndims, shapes_flat, partition_dims, R, T, home_of);
  if (rc != NS_OK) {
    delete pl;
    return rc;
  }
  make_mode_views(pl);
  *plan_out = pl;
  return NS_OK;
}

int ns_plan_create_flat(int n_tensors, const int32_t* ndims, const int64_t* shapes_flat, const int64_t* offsets,
                        int64_t buffer_size, const uint8_t* participating, int steps, float a, float b, float c,
                        float eps, int gram_mode, float ridge, int S, const int32_t* owner_of,
                        ns_plan_t** plan_out) {
  if (!plan_out) return NS_ERR_ARG;
  *plan_out = nullptr;
  if (n_tensors < 0 || (n_tensors > 0 && (!ndims || !shapes_flat || !offsets))) return NS_ERR_ARG;
  if (S < 1 || S > nsplan::kMaxRanks) return NS_ERR_ARG;
  int rc = check_coeffs(steps, eps, gram_mode, ridge);
  if (rc != NS_OK) return rc;
  ns_plan* pl = new (std::nothrow) ns_plan();
  if (!pl) return NS_ERR_ARG;
  Plan& p = pl->p;
  p.steps = steps;
  p.a = a;
  p.b = b;
  p.c = c;
  p.eps = eps;
  p.gram_mode = gram_mode;
  p.ridge = ridge;
  rc = nsplan::build_flat(p, n_tensors, ndims, shapes_flat, offsets, buffer_size, participating, S, owner_of);
  if (rc != NS_OK) {
    delete pl;
    return rc;
  }
  make_mode_views(pl);
  *plan_out = pl;
  return NS_OK;
}

int ns_plan_info(const ns_plan_t* plan, int64_t* info) {
  if (!plan || !info) return NS_ERR_ARG;
  const Plan& p = plan->p;
  info[0] = static_cast<int64_t>(p.t.size());
  info[1] = static_cast<int64_t>(p.part.size());
  info[2] = p.S;
  info[3] = p.layout;
  info[4] = p.gram_mode;
  info[5] = p.steps;
  info[6] = static_cast<int64_t>(p.buckets.size());
  info[7] = p.rank_len;
  info[8] = p.in_bytes;
  info[9] = p.out_bytes;
  return NS_OK;
}

int ns_plan_homes(const ns_plan_t* plan, int32_t* home_out) {
  if (!plan || (!home_out && !plan->p.t.empty())) return NS_ERR_ARG;
  for (size_t i = 0; i < plan->p.t.size(); ++i)
    home_out[i] = plan->p.t[i].participating ? plan->p.t[i].home : -1;
  return NS_OK;
}

int ns_plan_home_layout(const ns_plan_t* plan, int64_t* home_offsets, int64_t* home_sizes, int64_t* rank_sizes) {
  if (!plan) return NS_ERR_ARG;
  const Plan& p = plan->p;
  if (home_offsets)
    for (size_t i = 0; i < p.t.size(); ++i) home_offsets[i] = p.t[i].participating ? p.t[i].home_off : -1;
  if (home_sizes)
    for (int h = 0; h < p.S; ++h) home_sizes[h] = p.home_sizes[h];
  if (rank_sizes)
    for (int r = 0; r < p.S; ++r) rank_sizes[r] = p.rank_len;
  return NS_OK;
}

int ns_plan_workspace_bytes(const ns_plan_t* plan, uint64_t* bytes) {
  if (!plan || !bytes) return NS_ERR_ARG;
  *bytes = plan->p.ws_bytes;
  return NS_OK;
}

int ns_owner_gather_meta(const ns_plan_t* plan, int rho, int64_t* send_sizes, int64_t* recv_sizes,
                         int64_t* recv_offsets, int64_t* own_sizes) {
  if (!plan || plan->p.layout != NS_LAYOUT_FLAT || rho < 0 || rho >= plan->p.S) return NS_ERR_ARG;
  return nsplan::gather_meta(plan->p, rho, send_sizes, recv_sizes, recv_offsets, own_sizes);
}

int ns_owner_scatter_meta(const ns_plan_t* plan, int rho, int64_t* send_sizes, int64_t* recv_sizes,
                          int64_t* recv_offsets) {
  if (!plan || plan->p.layout != NS_LAYOUT_FLAT || rho < 0 || rho >= plan->p.S) return NS_ERR_ARG;
  return nsplan::scatter_meta(plan->p, rho, send_sizes, recv_sizes, recv_offsets);
}

// [LSA] route_to_ns_home as one all_to_allv, seen from rank rho (row-shard
// and two-stage plans). rho's send buffer holds, for each home h in rank
// order, rho's pieces of the tensors homed on h in index order; its receive
// buffer holds, for each source s in rank order, s's pieces of the tensors
// homed on rho in index order. route_from_ns_home is the same exchange with
// the send and receive sides swapped.
int ns_plan_rank_splits(const ns_plan_t* plan, int rho, int64_t* send_counts, int64_t* send_displs,
                        int64_t* recv_counts, int64_t* recv_displs, int64_t* send_pos, int64_t* recv_pos) {
  if (!plan || plan->p.layout == NS_LAYOUT_FLAT || rho < 0 || rho >= plan->p.S) return NS_ERR_ARG;
  const nsplan::Plan& p = plan->p;
  const int S = p.S;
  const size_t n = p.t.size();
  std::vector<int64_t> sc(S, 0), sd(S, 0);
  int64_t mine = 0;  // elements of one source's pieces of the tensors homed on rho
  for (size_t i = 0; i < n; ++i) {
    const nsplan::Tensor& t = p.t[i];
    if (!t.participating) continue;
    sc[t.home] += t.shard_len;
    if (t.home == rho) mine += t.shard_len;
  }
  for (int h = 1; h < S; ++h) sd[h] = sd[h - 1] + sc[h - 1];
  std::vector<int64_t> fill(sd);
  int64_t in_mine = 0;  // offset of a tensor's piece inside one source's segment
  for (size_t i = 0; i < n; ++i) {
    const nsplan::Tensor& t = p.t[i];
    const bool part = t.participating;
    if (send_pos) send_pos[i] = part ? fill[t.home] : -1;
    if (part) fill[t.home] += t.shard_len;
    for (int src = 0; src < S; ++src)
      if (recv_pos) recv_pos[i * S + src] = (part && t.home == rho) ? src * mine + in_mine : -1;
    if (part && t.home == rho) in_mine += t.shard_len;
  }
  for (int r = 0; r < S; ++r) {
    if (send_counts) send_counts[r] = sc[r];
    if (send_displs) send_displs[r] = sd[r];
    if (recv_counts) recv_counts[r] = mine;
    if (recv_displs) recv_displs[r] = r * mine;
  }
  return NS_OK;
}

const char* ns_status_string(int status) {
  switch (status) {
    case NS_OK: return "ok";
    case NS_ERR_ARG: return "invalid argument";
    case NS_ERR_SHAPE: return "invalid tensor shape (participating tensors need ndim >= 2)";
    case NS_ERR_NOT_DIVISIBLE: return "size not divisible by the number of ranks S";
    case NS_ERR_HOME: return "home/owner missing, out of range or not holding the tensor";
    case NS_ERR_CUDA: return "CUDA error";
    case NS_ERR_TIMEOUT: return "a kernel's bounded wait timed out";
    case NS_ERR_DEVICE_CHECK: return "a kernel refused an out-of-range index";
    case NS_ERR_UNSUPPORTED: return "not supported by this library or device";
    case NS_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
    default: return "unknown status";
  }
}

}  // extern "C"
