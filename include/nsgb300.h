/*
 * nsgb300 -- shape-batched quintic Newton-Schulz for GB300 (sm_103a), with the
 * shard -> home pack and home -> shard unpack around it.
 *
 * C ABI of libnsgb300.so. Every function returns an int status (NS_OK = 0 or
 * a negative NS_ERR_* code), never throws and never aborts the process.
 * Device buffers are plain device pointers owned by the caller; the library
 * owns only the plan (host metadata plus, for pack/unpack, a small device
 * routing table it allocates on the first pack/unpack call on a device).
 * Asynchronous work is ordered on the `stream` argument (a cudaStream_t passed
 * as void*; NULL = the legacy default stream). Errors found on the device
 * (a bounded wait that ran out, an index a kernel refused) are recorded in a
 * device status word and reported by ns_check_status().
 *
 * Sources (page title, entry):
 *  [LSA]  Megatron-Core API, core.optimizer.layer_sharded_a2a:
 *         params_by_home, route_to_ns_home, route_from_ns_home.
 *  [OP]   Megatron-Core API, core.distributed.fsdp.src.megatron_fsdp.
 *         experimental.owner_planning: select_ge_2d_params, ns_cost_fn,
 *         _OwnerWork, assign_owner_work, GroupOwnerLayout, OwnerGatherPlan,
 *         OwnerScatterPlan.
 *  [ISS]  Megatron-LM issue #6720 "[GTP][Muon] Optimize Muon step
 *         performance": shape-batched NS, SYRK symmetric kernels,
 *         fp32/TF32 Gram + trace ridge.
 */
#ifndef NSGB300_H
#define NSGB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------ status codes */
enum {
  NS_OK = 0,
  NS_ERR_ARG = -1,           /* null pointer, bad count, S/shard_dim mismatch   */
  NS_ERR_SHAPE = -2,         /* ndim < 2 for a participating tensor, bad dims   */
  NS_ERR_NOT_DIVISIBLE = -3, /* shard_dim size (or buffer size) not divisible by S */
  NS_ERR_HOME = -4,          /* home/owner missing, out of range, or not a holder */
  NS_ERR_CUDA = -5,          /* a CUDA runtime/driver call failed               */
  NS_ERR_TIMEOUT = -6,       /* a kernel's bounded wait ran out (device status)  */
  NS_ERR_DEVICE_CHECK = -7,  /* a kernel refused an out-of-range index           */
  NS_ERR_UNSUPPORTED = -8,   /* mode or device not supported by this library    */
  NS_ERR_WORKSPACE = -9      /* workspace missing, too small or misaligned       */
};

/* Precision policy of a plan (gram_mode). */
enum {
  NS_BF16 = 0,      /* bf16 X, A, B operands, fp32 accumulation and epilogues; bf16 in, bf16 out */
  NS_FP32_GRAM = 1, /* fp32 X, A, B as split-TF32 (hi, lo) pairs; bf16 in, fp32 out */
  /* [ISS] Gram-space NS ("gram_once"), same fp32 precision: A = X X^T once, then
   * per step Q = aI + bA + cA^2, A <- Q A Q, P <- Q P on m x m matrices only,
   * and X_k = P X_0 at the end. Exact reformulation of the same iteration;
   * fewer flops when n is well above m. bf16 in, fp32 out. */
  NS_FP32_GRAM_SPACE = 2,
  /* Per shape bucket, Gram-space when n >= 2m and NS_FP32_GRAM otherwise:
   * with k = 5 steps Gram-space does 4m^2n + 8km^3 flops against the
   * standard k(4m^2n + 2m^3), fewer once n > 1.875 m. Same precision and
   * results per matrix as the mode chosen for its bucket. bf16 in, fp32 out. */
  NS_FP32_AUTO = 3
};

/* Data model of a plan. */
enum {
  NS_LAYOUT_ROW_SHARD = 0, /* [LSA] every rank holds a (P/S, Q) slice of every param    */
  NS_LAYOUT_FLAT = 1,      /* [OP]  one flat buffer split evenly into S rank ranges     */
  NS_LAYOUT_TWO_STAGE = 2  /* [LSA] GTP_remat (dim 0) x TP (partition_dim) shards, one fused gather */
};

typedef struct ns_plan ns_plan_t; /* opaque; owned by the library */

/* ------------------------------------------------------------- host only */

/* [OP] ns_cost_fn. View `shape` (ndim >= 2) as (rows, cols) = (shape[0],
 * prod(shape[1:])); cost = rows*cols*(min(rows, cols)*steps + 1), exact in
 * int64. NS_ERR_SHAPE if ndim < 2 or a dim is negative; NS_ERR_ARG on null
 * pointers, steps < 0, or int64 overflow. */
int ns_cost(const int64_t* shape, int ndim, int steps, int64_t* cost_out);

/* [OP] assign_owner_work: greedy LPT. Tensors with one candidate are taken
 * first in index order, then the rest in descending cost (equal costs keep
 * index order); each goes to its least-loaded candidate, equal loads to the
 * candidate listed first. Candidates of tensor i are
 * cand_idx[cand_ptr[i] .. cand_ptr[i+1]) (CSR), ranks in [0, n_ranks), listed
 * in buffer order. owner_out[i] receives the owner. NS_ERR_HOME if a tensor
 * has no candidate or a candidate is out of range; NS_ERR_ARG on bad
 * arguments (costs must be > 0). */
int ns_assign_owner_work(int n_tensors, const int64_t* costs, const int32_t* cand_ptr,
                         const int32_t* cand_idx, int n_ranks, int32_t* owner_out);

/* [LSA] route_to_ns_home / route_from_ns_home plan cache, [OP] ns_cost_fn.
 * Row-shard plan over n_tensors params; tensor i has ndims[i] dims, listed
 * consecutively in shapes_flat. Every param is sharded S ways along
 * shard_dim (its size there must be divisible by S: NS_ERR_NOT_DIVISIBLE).
 * home_of[i] in [0, S) is param i's NS home; NULL asks for LPT homes over all
 * S ranks with cost ns_cost(shape, steps). steps >= 0; (a, b, c) are the
 * quintic coefficients used in every step; eps is added to the Frobenius
 * norm; ridge >= 0 adds ridge*(trace(A)/m)*I to A before B is formed (only
 * in NS_FP32_GRAM mode; must be 0 in NS_BF16 mode). The plan copies every
 * input array; the caller owns its validity only in the sense of [LSA]:
 * reuse it only while shapes, homes and S are unchanged. No CUDA call. */
int ns_plan_create(int n_tensors, const int32_t* ndims, const int64_t* shapes_flat, int steps,
                   float a, float b, float c, float eps, int gram_mode, float ridge, int S,
                   int shard_dim, const int32_t* home_of, ns_plan_t** plan_out);

/* [LSA] two-stage exchange (GTP_remat group along dim 0, then TP group along
 * partition_dim) and [ISS] its fusion into one exchange. S = R * T simulated
 * ranks, rank r*T + t holding remat slice r (along dim 0, of R) of TP slice t
 * (along partition_dims[i], of T) of every param, params in index order.
 * ns_pack_to_home assembles each param on its home in ONE gather, equal bit
 * for bit to running the two stages one after the other; ns_unpack_from_home
 * is its inverse. partition_dims[i] = 0 needs shape[0] % (R*T) == 0; else
 * shape[0] % R == 0 and shape[partition_dim] % T == 0 (NS_ERR_NOT_DIVISIBLE).
 * home_of in [0, R*T) or NULL for LPT homes. Other arguments as in
 * ns_plan_create. No CUDA call. */
int ns_plan_create_two_stage(int n_tensors, const int32_t* ndims, const int64_t* shapes_flat,
                             const int32_t* partition_dims, int R, int T, int steps, float a, float b,
                             float c, float eps, int gram_mode, float ridge, const int32_t* home_of,
                             ns_plan_t** plan_out);

/* [OP] GroupOwnerLayout / OwnerGatherPlan data model. Flat-buffer plan: tensor
 * i occupies elements [offsets[i], offsets[i] + numel_i) of a buffer of
 * buffer_size elements (buffer_size % S == 0, else NS_ERR_NOT_DIVISIBLE);
 * rank r holds [r*size/S, (r+1)*size/S). participating[i] != 0 marks the
 * tensors that take part (NULL = every tensor with ndim >= 2, the
 * select_ge_2d_params default); participating tensors must not overlap and
 * must have ndim >= 2 and numel > 0. owner_of[i] (read for participating i
 * only) must be a rank holding part of tensor i (NS_ERR_HOME otherwise);
 * NULL asks for assign_owner_work's default LPT owners. Other arguments as
 * in ns_plan_create. No CUDA call. */
int ns_plan_create_flat(int n_tensors, const int32_t* ndims, const int64_t* shapes_flat,
                        const int64_t* offsets, int64_t buffer_size, const uint8_t* participating,
                        int steps, float a, float b, float c, float eps, int gram_mode, float ridge,
                        int S, const int32_t* owner_of, ns_plan_t** plan_out);

/* Frees the plan and any device routing tables it uploaded. NULL is a no-op. */
int ns_plan_destroy(ns_plan_t* plan);

/* Plan summary: info[0] = n_tensors, [1] = participating count, [2] = S,
 * [3] = layout, [4] = gram_mode, [5] = steps, [6] = number of shape
 * buckets, [7] = per-rank buffer elements (row-shard) or buffer_size/S (flat),
 * [8] = input element bytes, [9] = output element bytes. info has >= 10 slots. */
int ns_plan_info(const ns_plan_t* plan, int64_t* info);

/* [LSA] params_by_home source: home_out[i] = home (owner) of tensor i, or -1
 * for a tensor that does not participate. home_out has n_tensors slots. */
int ns_plan_homes(const ns_plan_t* plan, int32_t* home_out);

/* Layout of the home buffers: home_offsets[i] = element offset of tensor i in
 * its home buffer (-1 if not participating); home_sizes[h] = elements in home
 * buffer h; rank_sizes[r] = elements in rank buffer r. Any pointer may be
 * NULL. Home h holds its tensors complete, in increasing index order. */
int ns_plan_home_layout(const ns_plan_t* plan, int64_t* home_offsets, int64_t* home_sizes,
                        int64_t* rank_sizes);

/* Bytes of device workspace ns_orthogonalize_batched needs (256-byte
 * aligned base required). Zero when nothing participates. */
int ns_plan_workspace_bytes(const ns_plan_t* plan, uint64_t* bytes);

/* [OP] OwnerGatherPlan metadata seen from rank rho (flat plans only, else
 * NS_ERR_ARG). send_sizes[o] = elements rho sends to owner o (0 = absent,
 * always 0 for o == rho); recv_sizes[s] = elements rho receives from s;
 * recv_offsets[i*S + s] = offset of tensor i's piece inside s's buffer to rho
 * (-1 = absent); own_sizes[i] = elements of rho's own shard of tensor i if
 * rho owns i, else -1. Any output pointer may be NULL. */
int ns_owner_gather_meta(const ns_plan_t* plan, int rho, int64_t* send_sizes, int64_t* recv_sizes,
                         int64_t* recv_offsets, int64_t* own_sizes);

/* [OP] OwnerScatterPlan metadata seen from rank rho (flat plans only):
 * send_sizes[d] = result elements rho (as owner) sends to d; recv_sizes[o]
 * = elements rho receives from owner o; recv_offsets[i*S + o] = offset of
 * tensor i's result piece inside o's buffer to rho (-1 = absent). */
int ns_owner_scatter_meta(const ns_plan_t* plan, int rho, int64_t* send_sizes, int64_t* recv_sizes,
                          int64_t* recv_offsets);

/* [LSA] route_to_ns_home / route_from_ns_home as one all_to_allv of row
 * shards, seen from rank rho (row-shard and two-stage plans; flat plans use
 * ns_owner_gather_meta, NS_ERR_ARG here). Every rank holds a piece of
 * numel/S elements of every participating tensor.
 *   send_counts[h], send_displs[h]: elements rho sends to home h and their
 *     offset in rho's send buffer, which holds, home by home in rank order,
 *     rho's pieces of the tensors homed on h in index order;
 *   recv_counts[s], recv_displs[s]: elements rho receives from rank s and
 *     their offset in rho's receive buffer (source by source in rank order,
 *     each segment the pieces of the tensors homed on rho in index order);
 *   send_pos[i]: offset of rho's piece of tensor i in its send buffer (-1 if
 *     tensor i does not participate);
 *   recv_pos[i*S + s]: offset of rank s's piece of tensor i in rho's receive
 *     buffer (-1 unless rho is tensor i's home).
 * The reverse exchange (route_from_ns_home) swaps the send and receive
 * sides. Arrays of S (counts, displs), n_tensors (send_pos) and n_tensors*S
 * (recv_pos) entries; any pointer may be NULL. Host only. */
int ns_plan_rank_splits(const ns_plan_t* plan, int rho, int64_t* send_counts, int64_t* send_displs,
                        int64_t* recv_counts, int64_t* recv_displs, int64_t* send_pos, int64_t* recv_pos);

const char* ns_status_string(int status);

/* ----------------------------------------------------------------- device */

/* [OP] ns_cost_fn step, [ISS] shape-batched NS. Orthogonalises the n
 * participating tensors of the plan (n must equal the participating count),
 * in index order: in[j] / out[j] are device pointers to the j-th participating
 * tensor, contiguous row-major in its original shape (bf16 in; bf16 out in
 * NS_BF16 mode, fp32 out in NS_FP32_GRAM mode). out[j] == in[j] is allowed;
 * other overlaps are not. Each tensor is viewed as (shape[0], prod(shape[1:])),
 * transposed so rows <= cols, scaled by 1/(||X||_F + eps), run for `steps`
 * steps of A = X X^T; X = a X + (b A + c A A) X, transposed back and stored.
 * workspace must hold ns_plan_workspace_bytes() bytes, 256-byte aligned; it
 * is scratch (no contents kept between calls). Asynchronous on `stream`;
 * calls that share a workspace must not overlap on the GPU. After a first
 * call on a device (it looks up per-device state), the call may be captured
 * into a CUDA graph and replayed: it allocates, synchronises and queries
 * nothing; a replay reads the buffers' current contents. The library's kernels
 * are launched with programmatic stream serialization: each may start its
 * set-up while the previous kernel in the stream runs, and reads or writes no
 * data before that kernel has completed, so ordering with the caller's work
 * on `stream` is as for ordinary launches. */
int ns_orthogonalize_batched(ns_plan_t* plan, const void* const* in, void* const* out, int n,
                             void* workspace, uint64_t workspace_bytes, void* stream);

/* [LSA] route_to_ns_home, [OP] OwnerGatherPlan.pack + reconstruct_full.
 * Device-local gather over S simulated ranks (no collective): rank_bufs[r]
 * (S device pointers, input dtype) hold rank r's data -- row-shard plans: its
 * (P/S, Q) shard of every param, in index order; flat plans: elements
 * [r*size/S, (r+1)*size/S) of the flat buffer. home_bufs[h] (S pointers)
 * receive home h's complete tensors in increasing index order, at the offsets
 * ns_plan_home_layout reports. S and shard_dim must equal the plan's (flat
 * plans: shard_dim 0). Bit-exact copy. The first pack/unpack call on a device
 * uploads the plan's routing table (cudaMalloc + copy): make it before any
 * stream capture. */
int ns_pack_to_home(ns_plan_t* plan, const void* const* rank_bufs, int S, int shard_dim,
                    void* const* home_bufs, void* stream);

/* [LSA] route_from_ns_home, [OP] OwnerScatterPlan.pack + unpack. Inverse of
 * ns_pack_to_home on the output dtype: home_bufs[h] hold complete results,
 * rank_bufs[r] receive rank r's shard of every result (flat plans: only the
 * elements of participating tensors are written). */
int ns_unpack_from_home(ns_plan_t* plan, const void* const* home_bufs, int S, int shard_dim,
                        void* const* rank_bufs, void* stream);

/* [ISS] wave dispatch, single-GPU form. A pipeline splits the plan's
 * participating tensors (bf16 plans only, else NS_ERR_UNSUPPORTED) into at
 * most n_waves waves of consecutive tensors with balanced ns_cost (no wave
 * when no tensor participates; one wave when every shape bucket runs as one
 * CTA per matrix, see ns_set_small_path; n_waves < 1 is NS_ERR_ARG). The plan must
 * outlive the pipeline. ns_pipeline_run then performs pack ->
 * Newton-Schulz -> unpack for the whole plan, with the same results as
 * ns_pack_to_home + ns_orthogonalize_batched + ns_unpack_from_home. Work runs
 * on three streams owned by the pipeline: the pack and prologue of a wave
 * overlap the NS products of the previous wave, and the unpack of a wave
 * overlaps the next one. Buffers as in ns_pack_to_home / ns_unpack_from_home
 * (home_in receives the gathered inputs, home_out the results); for row-shard
 * plans with shard_dim 0, where every row of a tensor is contiguous in one
 * rank buffer, the prologue reads the rank buffers directly and the last B*X
 * launch of each wave writes the results straight into rank_out, so home_in
 * and home_out are left untouched (a wave whose last launch cannot address
 * all its matrices still stages its results in home_out). When every bucket
 * of such a plan runs as one CTA per matrix, the whole call is that one
 * launch, issued on `stream` itself. workspace
 * holds two wave workspaces (ns_pipeline_info), 256-byte aligned. The call
 * is ordered after prior work on `stream`, and later work on `stream` waits
 * for all of it. The first run on a device creates the pipeline's streams
 * and events: make it before any stream capture. Runs that overlap on the
 * GPU must not share a pipeline or a workspace. */
typedef struct ns_pipeline ns_pipeline_t;
int ns_pipeline_create(ns_plan_t* plan, int n_waves, ns_pipeline_t** pipeline_out);
int ns_pipeline_info(const ns_pipeline_t* pipeline, int* n_waves, uint64_t* workspace_bytes);
int ns_pipeline_run(ns_pipeline_t* pipeline, const void* const* rank_in, void* const* home_in,
                    void* const* home_out, void* const* rank_out, void* workspace, uint64_t workspace_bytes,
                    void* stream);
int ns_pipeline_destroy(ns_pipeline_t* pipeline);

/* Synchronises `stream`, then reads and clears the current device's status
 * word: NS_ERR_TIMEOUT or NS_ERR_DEVICE_CHECK if a kernel recorded one, else
 * NS_ERR_CUDA on a pending CUDA error, else NS_OK. plan may be NULL. */
int ns_check_status(ns_plan_t* plan, void* stream);

/* No counterpart on the pages: an addition for callers that cannot allocate
 * device memory when they orthogonalise (e.g. a plugin inside a host program
 * whose caching allocator owns the GPU's memory, or code that must not call
 * cudaMalloc after start-up). Same computation and arguments as
 * ns_orthogonalize_batched, but the scratch memory is a static device array
 * of NS_FIXED_WS_BYTES inside the library instead of a caller workspace.
 * Allocates nothing (no cudaMalloc, no cudaFree). Returns NS_ERR_WORKSPACE if
 * the plan needs more than NS_FIXED_WS_BYTES (see ns_plan_workspace_bytes).
 * The array exists once per GPU that loads the library and is held until the
 * process exits. When it is reserved depends on CUDA's module loading: under
 * lazy loading (the default) the first call on a device, which looks up the
 * array's device address (cudaGetSymbolAddress) with that device current,
 * loads the module holding it and so reserves the NS_FIXED_WS_BYTES then --
 * that first call can fail with NS_ERR_CUDA if the GPU is already full, so
 * make it at start-up (and before any stream capture); under eager loading
 * (CUDA_MODULE_LOADING=EAGER) every process that loads the library holds the
 * array from the start, whether or not it calls this function. Every call
 * shares the array and finds the previous call's contents there (the kernels
 * write every byte they read first), so calls that overlap on the GPU (e.g.
 * on two streams) race. */
#define NS_FIXED_WS_BYTES (64ull << 20)
int ns_orthogonalize_batched_fixed_ws(ns_plan_t* plan, const void* const* in, void* const* out, int n,
                                      void* stream);

/* ---------------------------------------------------------- test support
 * No counterpart on the pages: hooks with which tests drive the library's
 * device-side error paths without faulting or hanging the GPU. */

/* Arms the next bf16 GEMM launch of this process (any phase, any thread) to
 * stall: its TMA producer issues no copy, so its MMA issuer's first wait for
 * operands cannot complete; every wait of that launch is bounded by
 * wait_limit_ns (1e5 .. 1e10 ns, else NS_ERR_ARG), after which the kernel
 * records a timeout in the device status word and unwinds (nothing is in
 * flight: no copy or MMA was issued). The call that contains the launch
 * returns normally but its results are garbage; ns_check_status then reports
 * NS_ERR_TIMEOUT, and later calls run normally. One-shot. */
int ns_test_stall_next_gemm(uint64_t wait_limit_ns);

/* Sets the home index of tensor `tensor` in the plan's routing table (and in
 * every device copy already uploaded) to `home`, which may be out of range:
 * pack and unpack then refuse that tensor's entry (its data is not moved),
 * record the refusal in the device status word, and ns_check_status reports
 * NS_ERR_DEVICE_CHECK. Restore the plan's own home to undo. NS_ERR_ARG if
 * the tensor has no routing entry. Synchronous (cudaMemcpy). */
int ns_test_set_route_home(ns_plan_t* plan, int tensor, int home);

/* ------------------------------------------------------------ measurement
 * Not part of the pages' interface: support for measuring the kernels above.
 * Kernel kinds: 0 = Gram (X X^T), 1 = A*A with the b*A + c*A^2 epilogue,
 * 2 = B*X with the a*X epilogue, 3 = norm/scale/transpose prologue and
 * output store, 4 = pack/unpack, 5 = the last step's B*X launches, which also
 * store the results (to the caller's tensors or the rank buffers), 6 = the
 * whole iteration of small matrices, one CTA per matrix. Launch
 * counters are always on. When timing
 * is enabled, every launch is bracketed by two CUDA events recorded on the
 * stream it is launched on; ns_profile_read synchronises those events. */

/* Tuning: how the bf16 GEMM phases use the tensor cores. cl = 1: one CTA per
 * 128 x 256 tile (tcgen05 cta_group::1); cl = 3: clusters of two CTAs running
 * the 2-SM MMA (cta_group::2) on 256 x 256 tiles, each SM holding half of
 * each operand; cl = 0 (default) picks 3 for the Gram and A*A phases, and 3
 * for B*X when every bucket has an even number of 128-row tile rows (else 1):
 * the fastest measured per phase. The paired mode applies to launches whose
 * buckets all have at least two 128-row tile rows; others use 1. Any other
 * value is NS_ERR_ARG. Process-wide; all modes give bitwise-identical
 * results. */
int ns_set_gemm_cluster(int cl);

/* Tuning: bf16 shape buckets with m <= 128 and n <= 512 (m, n the short and
 * long side of the 2-D view) run, when enable = 1 (the default), as one CTA per
 * matrix that keeps X, A and B in shared memory and the products in TMEM for
 * the whole iteration: one launch instead of a prologue, 3*steps GEMM
 * launches and a store. enable = 0 sends them through the GEMM launches like
 * every other bucket. Same arithmetic (bf16 operands, fp32 accumulation and
 * epilogues); results agree to rounding, not bit for bit. Other values are
 * NS_ERR_ARG. Process-wide. */
int ns_set_small_path(int enable);

/* Tuning: how the bf16 path stores the symmetric matrices A = X X^T and
 * B = b A + c A^2 (SYRK: only the tiles that touch the upper triangle are
 * computed; [ISS], SYRK symmetric kernels).
 * Both tilings compute exactly the upper 256 x 256 pair blocks of each
 * m_pad x m_pad result, in full. mode = 0 (the default): only those blocks
 * are stored, and the products that read A or B (A*A, B*X) load the K-blocks
 * left of their rows' diagonal pair block from the stored transposed block
 * (MN-major). mode = 1: the symmetric products also write the transpose of
 * every block above the diagonal pair blocks (the mirror), and the readers
 * take rows only. Other values are NS_ERR_ARG. Process-wide; both modes give
 * bitwise-identical results (the same products in the same K order). */
int ns_set_symmetric_store(int mode);

/* enable != 0 turns per-launch event timing on, 0 off. Process-wide. */
int ns_profile_enable(int enable);

/* launches[7] (may be NULL) receives the launch count per kind and gpu_ms[7]
 * (may be NULL) the summed event time per kind since the last reset; reset
 * != 0 clears both afterwards. */
int ns_profile_read(int reset, int64_t* launches, double* gpu_ms);

#ifdef __cplusplus
}
#endif

#endif /* NSGB300_H */
