// Host-side plan: per-tensor views, homes, routing offsets, shape buckets and
// the workspace layout. Built once by ns_plan_create / ns_plan_create_flat
// (pure host code) and reused by every device call.
#pragma once

#include <cstdint>
#include <vector>

#include "kernels.h"

namespace nsplan {

constexpr int kMaxDims = 8;
constexpr int kMaxRanks = 64;
constexpr int kMaxDevices = 64;

struct Tensor {
  int ndim = 0;
  int64_t shape[kMaxDims] = {0};
  int64_t rows = 0, cols = 0, numel = 0;  // 2-D view (shape[0], prod(shape[1:]))
  int64_t m = 0, n = 0;                   // min / max of (rows, cols)
  bool transposed = false;                // rows > cols
  bool participating = false;
  int64_t cost = 0;
  int home = -1;         // NS home (row-shard) or owner (flat)
  int64_t home_off = -1; // element offset inside its home buffer
  int ordinal = -1;      // position among participating tensors
  int bucket = -1, slot = -1;
  // row-shard routing: tensor viewed as (pre, D, post), shard_dim = D
  int64_t pre = 1, D = 1, post = 1, shard_len = 0, rank_off = 0;
  // sharded models: run length, run stride and rank bases of a piece
  int64_t run = 0, stride = 0, mr = 0, mt = 0;
  // flat routing
  int64_t flat_off = 0;
};

struct Bucket {
  int64_t m = 0, n = 0, m_pad = 0, n_pad = 0;
  std::vector<int> members;  // tensor indices, increasing
  uint64_t off_x0 = 0, off_x1 = 0, off_a = 0, off_b = 0;  // workspace byte offsets
  uint64_t off_partial = 0;  // float partial sums: count * nchunks
  uint64_t off_scale = 0;    // float scale per member
  uint64_t off_coef = 0;     // fp32 Gram-space: 3 floats per member (Q coefficients)
  int64_t nchunks = 0;       // sum-of-squares chunks per matrix
  bool gram_space = false;   // fp32: run this bucket in Gram space (NS_FP32_GRAM_SPACE, or NS_FP32_AUTO with n >= 2m)
  bool small = false;        // bf16, m <= 128, n <= 512: may run as one CTA per matrix (small.cu)
};

struct Plan {
  int layout = 0, S = 1, shard_dim = 0, steps = 5, gram_mode = 0;
  int R = 1, T = 1;         // two-stage model: GTP_remat x TP ranks (S = R * T)
  float a = 0, b = 0, c = 0, eps = 0, ridge = 0;
  int64_t buffer_size = 0;  // flat model
  int64_t rank_len = 0;     // elements per rank buffer
  std::vector<Tensor> t;
  std::vector<int> part;    // participating tensor indices, increasing
  std::vector<Bucket> buckets;
  std::vector<int64_t> home_sizes;
  uint64_t ws_bytes = 0;
  int in_bytes = 2, out_bytes = 2;
  // device routing table (one per device, uploaded on first pack/unpack)
  std::vector<nsk::RouteEntry> route;
  void* d_route[kMaxDevices] = {nullptr};
};

// Row count of one sum-of-squares chunk (elements).
constexpr int64_t kSumsqChunk = 32768;

int build_row_shard(Plan& p, int n, const int32_t* ndims, const int64_t* shapes, int S, int shard_dim,
                    const int32_t* home_of);
int build_two_stage(Plan& p, int n, const int32_t* ndims, const int64_t* shapes, const int32_t* pdims, int R,
                    int T, const int32_t* home_of);
int build_flat(Plan& p, int n, const int32_t* ndims, const int64_t* shapes, const int64_t* offsets,
               int64_t size, const uint8_t* participating, int S, const int32_t* owner_of);
int lpt_assign(int n, const int64_t* costs, const int32_t* cand_ptr, const int32_t* cand_idx, int n_ranks,
               int32_t* owner_out);
int build_subplan(const Plan& base, const std::vector<int>& members, Plan& out);

}  // namespace nsplan

// The opaque handle behind ns_plan_t.
struct ns_plan {
  nsplan::Plan p;
  // NS_FP32_AUTO: the plan's standard-fp32 and Gram-space buckets as two
  // views (same tensors, ordinals and workspace offsets), built at creation
  nsplan::Plan view_std, view_gs;
};
