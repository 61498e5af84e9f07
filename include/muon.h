/*
 * muon.h - C ABI of libmuon.so, a GB300 (sm_103a) implementation of the per-step
 * update of the sharded Muon optimizer for 2-D weight matrices held in flat buffers.
 *
 * Sources (page title, section):
 *   [P1] "Add initial Muon+M-FSDPv2 implementation" (Megatron-LM pull request #6425):
 *        "What does this PR do?" (every parameter placed in flat shards; one owner rank
 *        orthogonalizes each sharded matrix; other parameters take the regular optimizer
 *        path) and the "Opt step" pseudocode, steps 1-6.
 *   [P2] "core.distributed.fsdp.src.megatron_fsdp.experimental.muon" (Megatron-Core
 *        API docs), class FsdpMuon: step(), _step_group(), _compute_momentum_inputs(),
 *        _orthogonalize_updates(), _apply_local_updates(), "Limitations".
 *
 * The pages delegate the Muon arithmetic to a base class they do not print.  This
 * library takes the standard reading: M <- mu*M + G; orthogonalization input G + mu*M
 * (Nesterov, with the updated M) or M; quintic Newton-Schulz with
 * (a, b, c) = (3.4445, -4.7750, 2.0315) on X/||X||_F, transposed so rows <= cols;
 * decoupled weight decay W*(1 - lr*wd); update W -= lr*sqrt(max(1, rows/cols))*O.
 *
 * Conventions shared by every entry point
 *   - Every call returns a muon_status.  Arguments are validated before anything is
 *     launched; on a non-OK status nothing was enqueued and muon_last_error() holds a
 *     message (thread-local).
 *   - Pointers named *_shards / flat_* are HOST arrays of n_shards DEVICE pointers, one
 *     per flat shard of length L (muon_layout_shard_len).  Shard s holds flat elements
 *     [s*L, (s+1)*L); the tail of the last shard is padding and is never read or written.
 *     n_shards = 1 is the unsharded flat buffer.  Each shard pointer must be 16-byte
 *     aligned.  The caller owns all device memory (parameters, gradients, momentum,
 *     workspace); the library owns only the layout handle and small device tables.
 *   - Work is enqueued on `stream` and the call returns without waiting.  Kernels that
 *     wait on the GPU (mbarrier pipelines) give every wait an iteration budget; when one
 *     runs out the kernel records MUON_ERR_TIMEOUT in a device word and exits cleanly.
 *     muon_check() synchronises the stream and reports (and clears) that word.
 *   - The first GPU call on a layout uploads its device tables on the current device and
 *     the first call with a given workspace pointer encodes its TMA descriptors; both
 *     are synchronous.  Make those first calls before any CUDA-graph capture, and keep
 *     using the same device.  A layout must not be used from two threads at once.
 */
#ifndef MUON_H
#define MUON_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MUON_ABI_VERSION 1
#define MUON_MAX_SHARDS 128

typedef enum muon_status {
  MUON_OK = 0,
  MUON_ERR_INVALID_ARG = 1,   /* bad shape, count, NULL pointer, out-of-range scalar   */
  MUON_ERR_ALIGNMENT = 2,     /* a device pointer is not 16-byte (or 1024-byte) aligned */
  MUON_ERR_CUDA = 3,          /* a CUDA runtime call failed (message has the error)    */
  MUON_ERR_TIMEOUT = 4,       /* a device-side wait ran out of its budget              */
  MUON_ERR_OOM = 5,           /* host or device table allocation failed                */
  MUON_ERR_UNSUPPORTED = 6,   /* no sm_103a device, or a size beyond the library limits */
  MUON_ERR_DEVICE_CHECK = 7   /* debug builds: a device-side range check of a table     */
                              /* entry failed; the work it drove was skipped            */
} muon_status;

typedef enum muon_ns_dtype {
  MUON_NS_BF16 = 0,  /* Newton-Schulz on tcgen05 tensor cores: bf16 operands, fp32 accumulate */
  MUON_NS_FP32 = 1,  /* Newton-Schulz in fp32 on the CUDA cores (the precision path)          */
  /* fp32-accurate Newton-Schulz on the tensor cores: every fp32 operand x is kept as three
   * bf16 parts h = bf16(x), m = bf16(x - h), l = bf16(x - h - m), and every product takes
   * six tcgen05 kind::f16 MMAs (hh + hm + mh + hl + lh + mm) accumulated in fp32, within
   * about 2^-26 of the exact product.  The workspace holds the three parts (6 bytes per
   * element of X, A and B).  No counterpart on the pages: a faster form of MUON_NS_FP32. */
  MUON_NS_SPLIT_FP32 = 2
} muon_ns_dtype;

typedef struct muon_layout muon_layout; /* opaque */

/* ---------------------------------------------------------------- layout (host only)
 * muon_layout_create: describe one flat buffer ([P1]: every parameter in flat shards;
 * [P2] FsdpMuon, one FSDP buffer = one parameter group).
 *   shapes     n_params (rows, cols) pairs, int64, in flat-buffer order.  Parameters are
 *              packed back to back with no padding; N = sum(rows*cols).
 *   is_matrix  n_params flags; 0 marks a non-Muon parameter (a vector, an embedding the
 *              caller excludes) whose bytes the step never touches ([P2] "Limitations":
 *              non-2-D parameters are skipped).  NULL means every parameter is a matrix.
 *   n_shards   1..MUON_MAX_SHARDS equal flat shards, L = ceil(N / n_shards).
 *   ns_dtype   a muon_ns_dtype.
 * Matrices need rows, cols >= 1 and at most 2^31-1 elements; non-matrix parameters need
 * rows*cols >= 0.  n_params = 0 gives an empty layout on which every step is a no-op.
 * Pure host work: no GPU is touched.  *out receives a handle freed by muon_layout_destroy.
 */
muon_status muon_layout_create(const int64_t* shapes, const uint8_t* is_matrix,
                               int32_t n_params, int32_t n_shards, int32_t ns_dtype,
                               muon_layout** out);
/* Frees the handle and its device tables (on the device they were uploaded to).  NULL is OK. */
muon_status muon_layout_destroy(muon_layout* layout);
/* N, the number of flat elements described by the layout. */
muon_status muon_layout_numel(const muon_layout* layout, int64_t* numel);
/* L = ceil(N / n_shards), the length in elements of every shard. */
muon_status muon_layout_shard_len(const muon_layout* layout, int64_t* shard_len);
/* Bytes of device workspace muon_step and friends need.  The caller allocates it (e.g. a
 * torch uint8 tensor), 1024-byte aligned, and passes the same pointer to every call. */
muon_status muon_layout_workspace_bytes(const muon_layout* layout, size_t* bytes);
/* Length in elements of the fp32 "full" layout used by muon_gather_full & co: every
 * matrix parameter, row-major, each starting at a multiple of 4 elements. */
muon_status muon_layout_full_numel(const muon_layout* layout, int64_t* numel);
/* offsets[i] = element offset of matrix parameter i in the full layout, -1 for a
 * non-matrix parameter.  offsets must hold n_params entries. */
muon_status muon_full_offsets(const muon_layout* layout, int64_t* offsets);

/* ---------------------------------------------------------------- the optimizer step
 * muon_step: one optimizer step over the whole layout ([P2] FsdpMuon.step/_step_group;
 * [P1] "Opt step" 1-6 with the owner emulated on this GPU as indexing); it runs
 * muon_compute_momentum_inputs then muon_orthogonalize_apply:
 *   1. M <- mu*M + G and the orthogonalization input X = G + mu*M (nesterov != 0) or M,
 *      written straight into per-matrix full matrices in the workspace (the gather);
 *   2. per matrix, Newton-Schulz for ns_steps (0..100) iterations;
 *   3. W <- W*(1 - lr*wd) - lr*sqrt(max(1, rows/cols))*O, read back in shard order (the
 *      scatter).  The decay of [P2] _compute_momentum_inputs is applied here, in the same
 *      pass as the update, since X never depends on W.
 * flat_params and flat_momentum are updated in place; flat_grads is only read.  Momentum
 * must be zero before the first step.  Non-matrix positions and shard padding are untouched.
 */
muon_status muon_step(float* const* flat_params, const float* const* flat_grads,
                      float* const* flat_momentum, const muon_layout* layout, void* workspace,
                      float lr, float wd, float mu, int32_t nesterov, int32_t ns_steps,
                      cudaStream_t stream);

/* ---------------------------------------------------------------- optimizer groups
 * [P2] _FsdpGroupAssignment.tensor_to_optimizer_group_index maps each tensor of an FSDP
 * group to an optimizer group (its own lr, weight decay, momentum).  The grouping is a
 * property of the layout; the groups' values come with every call.
 * muon_layout_set_groups: group_of[i] in 0..n_groups-1 for every matrix parameter i (host
 * array of n_params entries; entries of non-matrix parameters are ignored), 1 <= n_groups
 * <= 32.  All matrices start in group 0.  If the layout's tables are already on the GPU
 * they are refreshed synchronously; do not call it while a step of this layout runs. */
muon_status muon_layout_set_groups(muon_layout* layout, const int32_t* group_of,
                                   int32_t n_groups);

typedef struct muon_group_hparams {
  float lr;          /* learning rate */
  float wd;          /* decoupled weight decay (the factor is 1 - lr*wd) */
  float mu;          /* momentum coefficient */
  int32_t nesterov;  /* nonzero: orthogonalize G + mu*M, else M */
} muon_group_hparams;

/* muon_step with per-group hyper-parameters: groups is a host array of the layout's
 * n_groups entries; matrix i uses groups[group_of[i]].  Everything else as muon_step. */
muon_status muon_step_grouped(float* const* flat_params, const float* const* flat_grads,
                              float* const* flat_momentum, const muon_layout* layout,
                              void* workspace, const muon_group_hparams* groups, int32_t ns_steps,
                              cudaStream_t stream);

/* The three stages of muon_step, callable one by one (same arguments, same meaning).
 * [P2] _compute_momentum_inputs: momentum update, input build, gather, Frobenius norms. */
muon_status muon_compute_momentum_inputs(const float* const* flat_grads,
                                         float* const* flat_momentum,
                                         const muon_layout* layout, void* workspace, float mu,
                                         int32_t nesterov, cudaStream_t stream);
/* [P2] _orthogonalize_updates: Newton-Schulz of every gathered matrix, in the workspace. */
muon_status muon_orthogonalize_updates(const muon_layout* layout, void* workspace,
                                       int32_t ns_steps, cudaStream_t stream);
/* [P2] _apply_local_updates: decay + scaled update into the parameter shards (scatter).
 * ns_steps must match the value given to muon_orthogonalize_updates. */
muon_status muon_apply_local_updates(float* const* flat_params, const muon_layout* layout,
                                     void* workspace, float lr, float wd, int32_t ns_steps,
                                     cudaStream_t stream);

/* Stages 2 and 3 in one call (what muon_step runs after stage 1).  On a tensor-core layout
 * (bf16 or split fp32) with ns_steps >= 1 whose Newton-Schulz iteration carries at least
 * 20 TFLOP (3 m^2 n + m^3 per matrix), the last Update applies
 * W <- W*(1 - lr*wd) - lr*scale*O in its epilogue, from the fp32 O before it is rounded,
 * and the separate apply pass is skipped (the fused tail); otherwise it equals
 * muon_orthogonalize_updates + muon_apply_local_updates.  The environment variable
 * MUON_FUSED_TAIL=1 or 0, read when the layout's tables are prepared, pins the choice.
 * The rounded O is stored either way, so muon_export_update stays valid. */
muon_status muon_orthogonalize_apply(float* const* flat_params, const muon_layout* layout,
                                     void* workspace, float lr, float wd, int32_t ns_steps,
                                     cudaStream_t stream);

/* ---------------------------------------------------------------- owner assignment
 * [P1] "What does this PR do?": for each sharded matrix one owner that holds at least one
 * of its shards is picked, and "Opt step" step 3: the owner is picked heuristically
 * depending on orthogonalization compute cost ([P2] tensor_to_owner_rank, computed once).
 * muon_assign_owners plans this for a data-parallel group of n_shards ranks (rank r holds
 * shard r): matrices in decreasing Newton-Schulz cost 5*(3 m^2 n + m^3)*ns_steps/5, each to
 * the least-loaded rank among those holding a part of it (ties: lowest rank), so a matrix
 * inside one shard stays on the rank that holds it.  owner: host array of
 * n_params entries (-1 for non-matrix parameters); rank_cost: host array of n_shards flop
 * totals, or NULL.  Pure host work, deterministic, so every rank computes the same plan. */
muon_status muon_assign_owners(const muon_layout* layout, int32_t ns_steps, int32_t* owner,
                               double* rank_cost);

/* ---------------------------------------------------------------- owner exchange plan
 * [P1] "Opt step" step 3 gathers each sharded matrix's orthogonalization input on its
 * owner and step 5 sends the owner's update back to the ranks that hold its shards ([P2]
 * _FsdpGroupAssignment.tensor_to_owner_rank names that owner).  muon_exchange_plan lists
 * the data plane of that exchange for a group of n_shards ranks (rank r holds shard r):
 * every matrix parameter's flat range cut at shard edges into runs, each run moved from
 * its shard on src_rank to the parameter's place in the owner's packed buffer on
 * dst_rank (step 3), and back along the same run (step 5).  The packed buffer of a rank
 * holds the parameters it owns, row-major, back to back in parameter order, each starting
 * at a multiple of 4 elements; its parameters read there are the full matrices
 * muon_gather_full builds, and runs written back reproduce muon_scatter_updates.
 * Runs whose src_rank equals dst_rank are local copies.  Pure host work, deterministic.
 *   owner          host array of n_params owners (muon_assign_owners' output works);
 *                  entries of matrix parameters must lie in 0..n_shards-1, the others are
 *                  ignored.
 *   rank           the rank whose lists are wanted, 0..n_shards-1.
 *   sends          runs with src_rank == rank, ordered by (dst_rank, parameter, offset);
 *   recvs          runs with dst_rank == rank, ordered by (src_rank, parameter, offset).
 *                  For each pair of ranks the sender's and the receiver's lists hold the
 *                  same runs in the same order, so one message per peer can carry them
 *                  back to back.  Either array may be NULL (then only its count is
 *                  returned); otherwise *n_sends / *n_recvs give its capacity on entry
 *                  (MUON_ERR_INVALID_ARG if too small) and the count on return.
 *   owned_numel    receives the length of `rank`'s packed buffer (may be NULL).
 *   owned_offsets  NULL or n_params entries: each parameter's offset in its owner's packed
 *                  buffer (-1 for non-matrix parameters). */
typedef struct muon_xfer {
  int32_t param;      /* parameter index */
  int32_t src_rank;   /* rank (= shard index) whose shard holds the run */
  int32_t dst_rank;   /* the parameter's owner */
  int32_t pad_;
  int64_t shard_off;  /* element offset of the run in src_rank's shard */
  int64_t owner_off;  /* element offset of the run in dst_rank's packed buffer */
  int64_t len;        /* elements in the run */
} muon_xfer;
muon_status muon_exchange_plan(const muon_layout* layout, const int32_t* owner, int32_t rank,
                               muon_xfer* sends, int64_t* n_sends, muon_xfer* recvs,
                               int64_t* n_recvs, int64_t* owned_numel, int64_t* owned_offsets);

/* ---------------------------------------------------------------- owner gather / scatter
 * [P1] "Opt step" step 3 (gather on the owner) and step 5 (scatter from the owner) as
 * pure index maps between the shards and the fp32 full layout.  Bit copies.
 * muon_gather_full writes every matrix of the full layout (full: device, full_numel
 * floats); muon_scatter_updates writes the matrix positions of the shards and nothing else. */
muon_status muon_gather_full(const muon_layout* layout, const float* const* shards,
                             float* full, cudaStream_t stream);
muon_status muon_scatter_updates(const muon_layout* layout, const float* full,
                                 float* const* shards, cudaStream_t stream);

/* ---------------------------------------------------------------- full-matrix access
 * muon_orthogonalize_full: Newton-Schulz of caller-given full matrices (fp32 full layout,
 * device) into full_out (same layout), through the same kernels as muon_step.  Uses (and
 * overwrites) the workspace. */
muon_status muon_orthogonalize_full(const muon_layout* layout, void* workspace,
                                    const float* full_in, float* full_out, int32_t ns_steps,
                                    cudaStream_t stream);
/* Copy the orthogonalization input the last stage 1 wrote (as stored: bf16 or fp32,
 * before normalisation) into full_out, widened to fp32. */
muon_status muon_export_input(const muon_layout* layout, const void* workspace,
                              float* full_out, cudaStream_t stream);
/* Copy the update O of the last stage 2 (ns_steps as given there) into full_out, fp32. */
muon_status muon_export_update(const muon_layout* layout, const void* workspace,
                               int32_t ns_steps, float* full_out, cudaStream_t stream);

/* ---------------------------------------------------------------- allocation-free variant
 * muon_orthogonalize_full_noalloc: muon_orthogonalize_full without any device allocation.
 * The paper has no counterpart to this entry point.  It is for callers that cannot call
 * cudaMalloc, nor have the library call it, where the orthogonalization runs: a host
 * framework whose caching allocator owns the device memory pool, a latency-critical loop
 * that cannot afford the synchronisation cudaMalloc / cudaFree may imply, a plugin inside
 * a process where only the host application allocates device memory.
 *   layout    a layout created with ns_dtype = MUON_NS_FP32 (the fp32 CUDA-core path);
 *             the tensor-core layouts (bf16, split fp32) return MUON_ERR_UNSUPPORTED.
 *   full_in   device, fp32 full layout (muon_full_offsets), 16-byte aligned: the inputs.
 *   full_out  device, same layout, 16-byte aligned: receives the orthogonalized updates.
 * Everything else (the layout's device tables and the workspace) lives in one file-scope
 * device array of 32 MiB (33,554,432 bytes) that every GPU loading the library holds until
 * the process exits.  A layout whose tables plus workspace exceed it is rejected with
 * MUON_ERR_UNSUPPORTED and a message giving both sizes.  The call allocates no device
 * memory (no cudaMalloc, cudaFree or allocating library routine); it uses host memory for
 * planning and cudaMemcpyAsync into the array.  The first call on a device looks up the
 * array's device address (cudaGetSymbolAddress) and zeroes the error word kept at its
 * start, with that device current; make that first call before any stream capture.
 * All calls share the array and leave their data in it: calls that overlap on the GPU
 * (different streams or threads) race.  Results equal those
 * of muon_orthogonalize_full on an fp32 layout. */
muon_status muon_orthogonalize_full_noalloc(const muon_layout* layout, const float* full_in,
                                            float* full_out, int32_t ns_steps,
                                            cudaStream_t stream);

/* ---------------------------------------------------------------- status
 * Synchronises `stream`, then reports a device-side wait timeout recorded since the last
 * check (MUON_ERR_TIMEOUT, and clears it), a failed range check of a debug build
 * (MUON_ERR_DEVICE_CHECK, and clears it) or a CUDA error (MUON_ERR_CUDA). */
muon_status muon_check(cudaStream_t stream);
/* Message for the last non-OK status returned on this thread ("" if none). */
const char* muon_last_error(void);
/* MUON_ABI_VERSION of the loaded library. */
int32_t muon_abi_version(void);
/* Which Newton-Schulz kernel `layout` runs on the current device; prepares the layout's
 * device tables there first if no call has (as the first step would).  The pages have no
 * counterpart: it reports a choice this library makes, for tests and measurements.
 * *tile_shape: 1 = one CTA per 128 x 256 tile (tcgen05 cta_group::1); 2 = a 2-CTA cluster
 * per 256 x 256 tile (cta_group::2); 3 = a 2-CTA cluster per 256 x 512 tile (two
 * cta_group::2 MMAs of N = 256 per k-step).  The environment variable MUON_TC_KERNEL=1, 2
 * or 3 pins the shape for layouts prepared afterwards (any other value:
 * MUON_ERR_INVALID_ARG).
 * *units: CTAs (shape 1) or clusters per launch.  *persistent = 1: all phases of all
 * iterations in one launch; 0: one launch per phase.  All three are 0 on fp32 layouts and
 * layouts without matrices.  MUON_ERR_UNSUPPORTED if the device is not sm_103, or the
 * environment (MUON_TC_KERNEL) pins a shape the device cannot run. */
muon_status muon_layout_ns_kernel(const muon_layout* layout, int32_t* tile_shape, int32_t* units,
                                  int32_t* persistent);
/* Where muon_step, muon_step_grouped and muon_orthogonalize_apply apply the update to W
 * on the current device: *fused = 1 inside the last Newton-Schulz Update's epilogue (from
 * the fp32 O), 0 in a separate streaming pass after the last Update (the pass
 * muon_apply_local_updates runs).  Prepares the layout's device tables first, as
 * muon_layout_ns_kernel does.  Tensor-core layouts fuse when one iteration carries
 * >= 20 TFLOP (symmetric count, sum over matrices of 3 m^2 n + m^3); the environment
 * variable MUON_FUSED_TAIL=0 or 1 pins the choice for layouts prepared afterwards.  fp32
 * layouts and layouts without matrices report 0, and a call with ns_steps = 0 never fuses.
 * The pages have no counterpart: a choice this library makes, reported for measurements. */
muon_status muon_layout_fused_apply(const muon_layout* layout, int32_t* fused);
/* Self-test of the bounded-wait path: launches one block that waits on an mbarrier nobody
 * arrives on, with a budget of budget_cycles clock cycles (1..2^40).  The wait runs out,
 * the kernel records MUON_ERR_TIMEOUT and returns; a following muon_check reports it. */
muon_status muon_selftest_wait_timeout(int64_t budget_cycles, cudaStream_t stream);

/* ---------------------------------------------------------------- debug builds
 * A library built with -DMUON_DEBUG (muon_optimizer_step_gb300.csrc.build --debug, which
 * writes libmuon_debug.so) checks every table entry inside the kernels before the access
 * it drives: chunk records (matrix index, extent, shard index and offset of the first and
 * last element, non-null shard pointers), matrix records (shape, pitches, workspace
 * buffers inside the workspace, flat extent inside the shards) and tile records (matrix
 * index, origin on the tile grid and inside the output, reduction length).  A failed
 * check records MUON_ERR_DEVICE_CHECK in the device error word, the kernel skips that work
 * (the tensor-core kernels skip their whole launch) and later kernels return at once
 * until muon_check reports and clears it.  Nothing traps.  The pages have no counterpart.
 * muon_debug_build: 1 in a debug build, 0 otherwise.
 * muon_selftest_device_check: debug builds only (else MUON_ERR_UNSUPPORTED): runs the
 * gather kernel on a one-chunk table whose chunk is longer than its matrix, built in a
 * small buffer this call allocates (every access the chunk describes stays inside that
 * buffer, so nothing can fault).  It synchronises `stream`; the following muon_check
 * returns MUON_ERR_DEVICE_CHECK. */
int32_t muon_debug_build(void);
muon_status muon_selftest_device_check(cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* MUON_H */
