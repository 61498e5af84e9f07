// Host-side launchers of the kernels (one translation unit each) used by capi.cu.
#pragma once

#include <cuda_runtime.h>
#include <cuda.h>

#include <string>

#include "muon_internal.h"

namespace muon {

struct ShardPtrs;
struct ApplyArgs;
struct GroupParams;
struct DebugCtx;

// Tile shapes of the tcgen05 Newton-Schulz kernels (the values MUON_TC_KERNEL pins and
// muon_layout_ns_kernel reports).
constexpr int kShapeSingle = 1;  // one CTA per 128 x 256 tile, tcgen05 cta_group::1
constexpr int kShapePair = 2;    // 2-CTA cluster per 256 x 256 tile, tcgen05 cta_group::2
constexpr int kShapePairWide = 3;  // 2-CTA cluster per 256 x 512 tile: two cta_group::2
                                   // MMAs of N = 256 per k-step into one 512-column accumulator

// Device-resident tables of a layout (uploaded once per device).
struct DevTables {
  int device = -1;
  int n_sms = 0;
  ChunkDev* chunks = nullptr;
  MatDev* mats = nullptr;
  int* err = nullptr;           // device error word (MUON_ERR_TIMEOUT when a wait gave up)
  // fp32 path: one tile list per phase
  TileDev* tiles[3] = {nullptr, nullptr, nullptr};
  int32_t* cta_begin[3] = {nullptr, nullptr, nullptr};
  int64_t n_tiles[3] = {0, 0, 0};  // entries of each phase's tile list
  int grid[3] = {0, 0, 0};
  // Tensor-core paths: tc_lists tile lists back to back in tc_tiles; list l's offsets for
  // unit u are tc_begin[l * (tc_units + 1) + u] and the next entry.  One list per phase,
  // or, for a persistent launch, one per iteration and phase (q = 3 * it + phase), the
  // last iteration's lists serving any later one.
  TileDev* tc_tiles = nullptr;
  int32_t* tc_begin = nullptr;
  int tc_lists = 0;
  int64_t tc_n_tiles = 0;
  CUtensorMap* tmaps = nullptr; // kMapsPerMat per matrix (bf16 path)
  int tc_shape = kShapeSingle;  // bf16 path: tile shape (kShape*)
  bool tc_persistent = false;   // bf16 path: all phases in one launch
  bool fused_tail = false;      // tensor-core paths: the last Update applies W itself
  int tc_units = 0;             // tensor-core paths: CTAs (or pairs) of each launch
  const void* tmap_ws = nullptr;  // workspace the tensor maps were encoded for
};

// What the debug range checks of the kernels compare against (see DebugCtx).
DebugCtx make_debug_ctx(const Plan& plan, const DevTables& dt);

// Stage 1: momentum, orthogonalization input into X0, per-chunk sums of squares.
cudaError_t launch_momentum_input(const Plan& plan, const DevTables& dt, const ShardPtrs& g,
                                  const ShardPtrs& m, void* ws, const GroupParams& gp,
                                  cudaStream_t st);
// Full fp32 matrices -> X0 plus per-chunk sums of squares.
cudaError_t launch_full_input(const Plan& plan, const DevTables& dt, const float* full, void* ws,
                              cudaStream_t st);
// Per-matrix 1/||X||_F from the chunk sums (deterministic order).
cudaError_t launch_norm_finalize(const Plan& plan, const DevTables& dt, void* ws,
                                 cudaStream_t st);
// Stage 3: W <- W*decay - lr*scale*O, O read from the final X buffer.
cudaError_t launch_apply(const Plan& plan, const DevTables& dt, const ShardPtrs& w,
                         const void* ws, int final_buf, int pending_norm, const GroupParams& gp,
                         cudaStream_t st);
// Owner gather / scatter between shards and the fp32 full layout.
cudaError_t launch_gather(const Plan& plan, const DevTables& dt, const ShardPtrs& src,
                          float* full, cudaStream_t st);
cudaError_t launch_scatter(const Plan& plan, const DevTables& dt, const float* full,
                           const ShardPtrs& dst, cudaStream_t st);
// X buffer (0 or 1) -> fp32 full layout, times 1/||X|| when pending_norm.
cudaError_t launch_export(const Plan& plan, const DevTables& dt, const void* ws, int buf,
                          int pending_norm, float* full, cudaStream_t st);

// Stage 2, bf16 path: all ns_steps iterations of every matrix in one persistent tcgen05
// launch (with ap != nullptr the last Update also applies the step to the weights).
cudaError_t launch_ns_tc(const Plan& plan, const DevTables& dt, void* ws, int ns_steps,
                         long long budget, const ApplyArgs* ap, cudaStream_t st);
// Shared-memory opt-in of the tcgen05 kernels and how many CTA pairs / single CTAs can be
// resident at once.
cudaError_t prepare_ns_kernels(int* max_pairs, int* max_singles);
// Stage 2, fp32 path: one SIMT GEMM phase over every matrix.
cudaError_t launch_ns_phase_f32(const Plan& plan, const DevTables& dt, void* ws, int phase,
                                int x_in, int iter0, cudaStream_t st);
// Encodes the bf16 path's tensor maps for workspace `ws` into host memory.
bool encode_tensor_maps(const Plan& plan, const void* ws, std::vector<CUtensorMap>* maps,
                        std::string* err);
// One-block kernel that waits on an mbarrier nobody arrives on, with `budget` cycles.
cudaError_t launch_selftest_timeout(int* err, long long budget, cudaStream_t st);
// Sets the message muon_last_error() returns on this thread.
void set_last_error(const std::string& msg);
// The allocation-free entry point's error word on device `dev` (inside its scratch
// array), or nullptr if that entry point has not run there.
int* noalloc_error_word(int dev);

}  // namespace muon
