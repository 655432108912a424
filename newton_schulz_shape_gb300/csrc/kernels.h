// Launch parameters shared by the host orchestration (orchestrate.h) and the kernels
// (gemm.cu, prologue.cu, pack.cu), and the launcher entry points. Everything a
// kernel needs per call travels by value in its parameter block, so the
// Newton-Schulz path itself allocates nothing.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace nsk {

// ------------------------------------------------------------------- GEMMs
constexpr int GEMM_MAX_BUCKETS = 8;
constexpr int ROUTE_MAX_RANKS = 64;
enum GemmPhase { PH_GRAM = 0, PH_A2B = 1, PH_BX = 2 };

struct GemmBucket {
  long long tile_begin;  // first global tile index of this bucket
  long long out_stride;  // elements between consecutive matrices of `out`
  long long aux_stride;  // elements between consecutive matrices of `aux`
  void* out;             // bf16: A (Gram), B (A2B), X_next (BX)
  const void* aux;       // bf16: A (A2B), X_cur (BX), unused (Gram)
  int count;             // matrices in the bucket
  int tiles_m, tiles_n;  // tile grid of one output matrix
  int tiles_per_mat;     // tiles computed per matrix (upper ones only for SYRK)
  int k_blocks;          // K / 64
  int ld_out, ld_aux;    // leading dimensions (elements)
  int cols_valid;        // output columns that exist (m_pad or n_pad)
  int m_valid, n_valid;  // unpadded m, n (final-store launches)
  int out_first;         // first entry of this bucket in out_tab (final-store launches)
  const float* scale;    // first step's Gram and B*X: per-matrix 1 / (||T||_F + eps), X~_0
                         // being unscaled (Gram: out = s^2 acc; B*X: out = s (a aux + acc));
                         // null otherwise
};

// Final-store launches of the B*X phase write each result straight to the
// caller's output tensor; out_tab holds one entry per matrix: the output
// address with bit 0 set when the tensor was transposed (rows > cols). With
// out_ranks the results go straight to the S rank buffers instead (row
// shards along dim 0): the entry is the tensor's shard offset in every rank
// buffer (elements) shifted left by one, with the same bit 0.
constexpr int GEMM_MAX_OUT = 3312;

// A and B are stored as their upper 256 x 256 pair blocks only: block rows
// 256 Q .. 256 Q + 255, columns from 256 Q on, each block in full (the SYRK
// tiles compute exactly these). A product reading a symmetric operand takes
// the 64-wide K-blocks left of its rows' diagonal pair block (columns below
// 256 Q) from the transposed, stored block: the same values, loaded MN-major.
template <int NOUT>
struct GemmParamsT {
  CUtensorMap tma[GEMM_MAX_BUCKETS];  // A operand, K-major, box {64, 128, 1}
  CUtensorMap tmb[GEMM_MAX_BUCKETS];  // B operand: K-major box {64,128,1} (Gram) / MN-major box {64,64,1}
  CUtensorMap tmt[GEMM_MAX_BUCKETS];  // A operand MN-major, box {64, 64, 1} (A*A: A; B*X: B)
  // epilogue chunks, box {32, 32, 1}, 64-byte swizzle: aux (A2B: A, BX: X)
  // and output (final-store launches write from registers: no output map)
  CUtensorMap tme[GEMM_MAX_BUCKETS];
  CUtensorMap tmo[NOUT == 1 ? GEMM_MAX_BUCKETS : 1];
  GemmBucket bk[GEMM_MAX_BUCKETS];
  long long total_tiles;
  int nb;
  float alpha, beta, gamma;  // a, b, c of the quintic step
  int reverse;               // walk the tiles last to first (serpentine order across launches)
  int mirror;                // symmetric outputs also store their mirror; readers of A and B take rows only
  // Test support: wait_ns (0 = NS_WAIT_LIMIT_NS) bounds every mbarrier wait of
  // the launch; stall != 0 makes the TMA producer issue no copy at all, so the
  // MMA issuer's first wait for operands runs out after wait_ns and the
  // kernel unwinds with NS_DEV_TIMEOUT recorded (nothing is in flight then).
  unsigned long long wait_ns;
  int stall;
  int out_ranks;             // final-store launches: out_tab holds rank-buffer offsets
  int S;                     // ranks of rank_ptr (out_ranks)
  void* rank_ptr[ROUTE_MAX_RANKS];
  unsigned int* status;
  unsigned long long out_tab[NOUT];
};
using GemmParams = GemmParamsT<1>;
using GemmFinalParams = GemmParamsT<GEMM_MAX_OUT>;
static_assert(sizeof(GemmFinalParams) <= 32764, "kernel parameter block too large");

constexpr int GEMM_BM = 128, GEMM_BN = 256, GEMM_BK = 64;

// ----------------------------------------------------- fp32-Gram GEMMs
enum Gemm32Phase { PH32_GRAM = 0, PH32_A2B = 1, PH32_BXT = 2 };

struct Gemm32Bucket {
  long long tile_begin;
  long long mat_stride;    // elements between matrices of the m-major buffers (A, B or X)
  long long mat_stride_t;  // elements between matrices of the transposed X buffers
  float* out_h;            // Gram: A hi; A2B: B hi; BXT: next X hi (m_pad x n_pad)
  float* out_l;
  float* out_th;           // BXT: next X^T hi (n_pad x m_pad)
  float* out_tl;
  const float* aux_h;      // A2B: A hi (may be null: no aux term); BXT: current X hi
  const float* aux_l;
  const float* coef;       // A2B: per-matrix (delta, beta, gamma) or null (use delta/beta/gamma below)
  float delta, beta, gamma;  // A2B: out = delta*I + beta*aux + gamma*acc when coef is null
  int count, tiles_m, tiles_n, tiles_per_mat, k_blocks;
  int ld;                  // leading dimension of out_h/out_l/aux (elements)
  int ld_t;                // leading dimension of out_th/out_tl
  int cols_valid;          // tile columns that exist (m_pad)
  int m_valid, n_valid;    // unpadded m, n (final-store launches)
  int out_first;
};

constexpr int GEMM32_MAX_OUT = 3200;
// K block of the fp32 kernels: 16 fp32 (64-byte rows, 64-byte swizzle), so
// that a stage (hi and lo of a 128-row A tile and a 256-row B tile) is 48 KB
// and four stages fit in shared memory
constexpr int GEMM32_BK = 16;

template <int NOUT>
struct Gemm32ParamsT {
  CUtensorMap tmah[GEMM_MAX_BUCKETS];  // A operand hi / lo, K-major, box {32, 128, 1} fp32
  CUtensorMap tmal[GEMM_MAX_BUCKETS];
  CUtensorMap tmbh[GEMM_MAX_BUCKETS];  // B operand hi / lo, K-major, box {32, 128, 1} fp32
  CUtensorMap tmbl[GEMM_MAX_BUCKETS];
  Gemm32Bucket bk[GEMM_MAX_BUCKETS];
  long long total_tiles;
  int nb;
  int pair;            // 2-SM form: work items are pairs of 128-row tiles (rows 2q, 2q + 1)
  float alpha, beta, gamma;
  unsigned int* status;
  unsigned long long out_tab[NOUT];
};
using Gemm32Params = Gemm32ParamsT<1>;
using Gemm32FinalParams = Gemm32ParamsT<GEMM32_MAX_OUT>;
static_assert(sizeof(Gemm32FinalParams) <= 32764, "kernel parameter block too large");

struct Ridge32Bucket {
  float* ah;
  float* al;
  long long mat_stride;
  int ld, m, count;
};

struct Ridge32Params {
  Ridge32Bucket bk[GEMM_MAX_BUCKETS];
  int nb, max_count;
  float ridge;
  float a, b, c;          // Gram-space coefficients: writes coef = (a + b r + c r^2, b + 2 c r, c)
  float* coef[GEMM_MAX_BUCKETS];  // null: add the ridge to A's diagonal instead
};

// ------------------------------------------------------- prologue / store
constexpr int PRO_MAX_MATS = 192;

struct MatDesc {
  const void* in;       // original tensor, row-major (rows x cols), bf16
  void* out;            // result, row-major (rows x cols)
  void* x;              // this matrix's X_0 in the workspace (m_pad x n_pad, bf16;
                        // fp32-Gram: X hi, with X lo, X^T hi, X^T lo at x_split apart)
  const void* xfinal;   // this matrix's X_k in the workspace (fp32-Gram: X hi; X lo at x_split)
  float* partial;       // nchunks partial sums of squares
  float* scale;         // 1 / (||X||_F + eps)
  long long numel;
  int rows, cols;
  int transposed;
  long long rank_off;   // rank-buffer input (ProParams.from_ranks): element offset of this tensor's
                        // shard in every rank buffer; row j of the tensor is row j % shard_rows of
                        // the shard on rank j / shard_rows
  int shard_rows;
};

struct ProParams {
  MatDesc md[PRO_MAX_MATS];
  int count;
  int nchunks;          // sum-of-squares chunks per matrix (same for the batch)
  int m_pad, n_pad;     // workspace matrix dims (same for the batch)
  int m, n;             // valid dims after the transpose
  float eps;
  int out_f32;          // result dtype: 0 bf16, 1 fp32
  long long x_split;    // fp32-Gram: elements between the X hi / X lo / X^T hi / X^T lo buffers
  int apply_scale;      // store: multiply by *scale (bf16 path with zero steps)
  int from_ranks;       // bf16 prep: read the tensors' rows from the rank buffers (row shards along
                        // dim 0) instead of md[].in: the pack to the home buffer is fused away
  int ranks_aligned;    // every rank_ptr is 16-byte aligned
  const void* rank_ptr[ROUTE_MAX_RANKS];
  unsigned int* status;
};

// ----------------------------------------------------------- pack / unpack

struct RouteEntry {
  long long seg_begin;  // first position of the tensor in the rank coordinate space
  long long seg_len;    // positions it occupies there
  long long home_off;   // element offset of the complete tensor in its home buffer
  long long inner;      // sharded models: contiguous run inside a rank's piece
  long long outer;      // sharded models: stride between runs in the full tensor
  long long mr, mt;     // sharded models: rank rho = r * T + t starts its piece at
                        // r * mr + t * mt of the full tensor (row-shard: T = 1)
  int home;
  int pad;
};

struct PackParams {
  void* rank_ptr[ROUTE_MAX_RANKS];
  void* home_ptr[ROUTE_MAX_RANKS];
  const RouteEntry* entries;
  long long n_entries;
  long long rank_len;   // positions per rank buffer
  long long chunk;      // positions per CTA
  long long g_begin;    // entry-coordinate range to move (a wave of the pipeline, or everything)
  long long g_end;
  int S;
  int T;                // TP ranks of the two-stage model (1 otherwise)
  int flat;             // 1: flat-buffer model, 0: row-shard / two-stage model
  int elem_bytes;       // 2 or 4
  int to_home;          // 1: pack (rank -> home), 0: unpack (home -> rank)
  unsigned int* status;
};

// ------------------------------------------------- small matrices, one CTA each
// m <= 128 and n <= SMALL_MAX_N: the whole iteration of one matrix runs in
// one CTA (small.cu), from the input tensor to the result.
constexpr int SMALL_MAX_M = 128;
constexpr int SMALL_MAX_N = 512;
constexpr int SMALL_MAX_MATS = 512;

struct SmallMat {
  const void* in;      // tensor, row-major rows x cols, bf16 (unused with in_ranks)
  void* out;           // result, same shape (unused with out_ranks)
  long long rank_off;  // rank-buffer modes: the tensor's shard offset (elements) in every rank buffer
  int rows, cols;      // 2-D view (shape[0], prod(shape[1:]))
  int transposed;      // rows > cols
  int pad;
};

// The per-matrix table comes last and is sized per launch (the launcher
// copies a table of up to N entries into the smallest block that holds it:
// a large parameter block costs launch time).
template <int N>
struct SmallParamsT {
  int count;
  int n_pad;           // largest n rounded up to 64 over the launch (sizes smem and TMEM)
  int steps;
  float a, b, c, eps;
  int S;               // rank buffers of the rank modes
  int in_ranks;        // read row j of a tensor from rank j / (rows / S) (row shards along dim 0)
  int out_ranks;       // write the result rows the same way
  const void* rank_in[ROUTE_MAX_RANKS];
  void* rank_out[ROUTE_MAX_RANKS];
  unsigned int* status;
  SmallMat mat[N];
};
using SmallParams = SmallParamsT<SMALL_MAX_MATS>;
static_assert(sizeof(SmallParams) <= 32764, "kernel parameter block too large");

// ----------------------------------------------------------------- launchers
// 1-SM form: one CTA per 128 x 256 tile. The launchers size the grid from
// the work items, the SM count and cluster occupancy.
cudaError_t launch_gemm(int phase, const GemmParams& p, int nsm, cudaStream_t st);
cudaError_t launch_gemm_final(const GemmFinalParams& p, int nsm, cudaStream_t st);
// 2-SM form (tcgen05 cta_group::2): clusters of two CTAs compute 256 x 256
// tiles; p.bk[].tiles_per_mat counts tile-row pairs.
cudaError_t launch_gemm_pair(int phase, const GemmParams& p, int nsm, cudaStream_t st);
cudaError_t launch_gemm_pair_final(const GemmFinalParams& p, int nsm, cudaStream_t st);
cudaError_t launch_sumsq(const ProParams& p, cudaStream_t st);
cudaError_t launch_scale(const ProParams& p, cudaStream_t st);
cudaError_t launch_prep(const ProParams& p, cudaStream_t st);
cudaError_t launch_store(const ProParams& p, cudaStream_t st);
cudaError_t launch_pack(const PackParams& p, cudaStream_t st);
// fp32 split-TF32 GEMMs; p.pair selects the 2-SM form (clusters of two CTAs,
// tcgen05 cta_group::2), which needs every bucket to have >= 2 tile rows.
cudaError_t launch_gemm32(int phase, const Gemm32Params& p, int nsm, cudaStream_t st);
cudaError_t launch_gemm32_final(const Gemm32FinalParams& p, int nsm, cudaStream_t st);
cudaError_t launch_ridge32(const Ridge32Params& p, cudaStream_t st);
cudaError_t launch_prep32(const ProParams& p, cudaStream_t st);
cudaError_t launch_store32(const ProParams& p, cudaStream_t st);
cudaError_t launch_small(const SmallParams& p, cudaStream_t st);

}  // namespace nsk
