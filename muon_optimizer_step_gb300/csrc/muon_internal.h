// Internal data structures shared by the host planner (layout.cpp), the C ABI
// (capi.cu) and the kernels.  Plain structs only, so that g++ and nvcc agree on them.
#pragma once

#include <cstddef>
#include <cstdint>
#include <string>
#include <vector>

namespace muon {

// Flat elements handled by one entry of the chunk table.  A chunk never crosses a
// matrix boundary; it starts at a multiple of kChunkElems of the matrix's row-major
// index.  One that lies inside one shard (the usual case) is read through that shard's
// pointer with 128-bit loads; one that crosses a shard edge is read element by element.
constexpr int kChunkElems = 32768;

// Workspace alignment of every per-matrix buffer (TMA wants 16 B; SW128 tiles 1024 B).
constexpr int64_t kWsAlign = 1024;

// Optimizer groups whose hyper-parameters a call can carry (by value, in kernel arguments).
constexpr int kMaxGroups = 32;

// tcgen05 NS tile (bf16 path) and SIMT NS tile (fp32 path).
constexpr int kTcBM = 128;
constexpr int kTcBN = 256;
constexpr int kTcBK = 64;
constexpr int kF32BM = 128;
constexpr int kF32BN = 128;

// Tensor maps per matrix on the tensor-core paths (index = mat * kMapsPerMat + slot).
enum MapSlot {
  kMapX0K128 = 0, kMapX0K256 = 1, kMapX0MN = 2,
  kMapX1K128 = 3, kMapX1K256 = 4, kMapX1MN = 5,
  kMapAK128 = 6, kMapAK256 = 7,
  kMapBK128 = 8, kMapBK256 = 9,
  // bf16: 32 x 32 boxes with 64-byte swizzle for the epilogue's TMA stores
  kMapX0St = 10, kMapX1St = 11, kMapASt = 12, kMapBSt = 13,
  // split fp32: slots 0-9 map the h arrays, slot + kMapPart the m, + 2 kMapPart the l
  kMapPart = 14,
  kMapsPerMat = 42
};

enum Phase { kPhaseGram = 0, kPhasePoly = 1, kPhaseUpdate = 2 };

struct ChunkDev {          // 32 bytes
  int32_t mat;             // matrix index (dense, over matrix parameters only)
  int32_t shard;           // shard holding the chunk's first element
  int64_t shard_off;       // its offset inside that shard
  int64_t local;           // row-major element index inside the matrix
  int32_t len;             // elements in the chunk
  int32_t vec;             // 1: inside one shard, and offsets allow 128-bit accesses
};

struct MatDev {            // 120 bytes
  int32_t rows, cols;      // stored shape
  int32_t m, n;            // min / max of (rows, cols)
  int32_t tall;            // rows > cols: work on X^T (A = X^T X, X' = aX + X B)
  int32_t ldx;             // row pitch (elements) of the X buffers
  int32_t lda;             // row pitch (elements) of the A and B buffers (m x m)
  int32_t param;           // index of the parameter in the caller's shapes list
  int64_t x0, x1, a, b;    // byte offsets in the workspace
  int64_t full_off;        // element offset in the fp32 full layout
  int64_t chunk_begin;     // chunk table range of this matrix
  int64_t chunk_end;
  float scale;             // sqrt(max(1, rows/cols))
  int32_t group;           // optimizer group (index into per-call hyper-parameters)
  int64_t flat_off;        // element offset of the matrix in the unsharded flat buffer
  int32_t sig[3];          // per phase: CTA-tiles that signal completion (tcgen05 path)
  int32_t pad2_;
};

struct TileDev {           // 16 bytes: one output tile of one GEMM phase
  int32_t mat;
  int32_t i0, j0;          // first row / column of the tile in the phase's output
  int32_t kblocks;         // ceil(K / BK): reduction length in k-blocks
};

// A per-phase work list: tiles ordered CTA by CTA, cta_begin has grid+1 entries.
struct TileList {
  std::vector<TileDev> tiles;
  std::vector<int32_t> cta_begin;
  int grid = 0;
};

// Host-side plan of one flat buffer (everything that needs no GPU).
struct Plan {
  int32_t n_params = 0;
  int32_t n_shards = 1;
  int32_t ns_dtype = 0;               // 0 bf16, 1 fp32, 2 split fp32 (bf16 x 3)
  int64_t N = 0;                      // flat elements
  int64_t L = 0;                      // shard length
  int64_t full_numel = 0;
  std::vector<int64_t> rows, cols;    // per parameter
  std::vector<uint8_t> is_matrix;
  std::vector<int64_t> flat_off;      // per parameter
  std::vector<int64_t> full_off;      // per parameter, -1 for non-matrix
  int32_t n_groups = 1;               // optimizer groups (muon_layout_set_groups)
  std::vector<MatDev> mats;           // matrix parameters with numel > 0
  std::vector<ChunkDev> chunks;
  // Workspace: [partials: n_chunks f32][inv_norm: n_mats f32][counters: 3 n_mats i32]
  //            [per-matrix buffers]
  int64_t ws_partials = 0;
  int64_t ws_inv_norm = 0;
  int64_t ws_counters = 0;            // per matrix and phase: finished tiles (int32)
  int64_t ws_bytes = 0;
};

// Returns "" on success, else a message.  Pure host arithmetic.
std::string build_plan(const int64_t* shapes, const uint8_t* is_matrix, int32_t n_params,
                       int32_t n_shards, int32_t ns_dtype, Plan* plan);

// Assignment of a phase's tiles to `grid` CTAs (grid <= n_sms), each tile to the least
// loaded CTA: longest first (by_cost), or in matrix order.  One launch per phase uses the
// first; a persistent launch plans its lists with plan_persistent instead.
TileList plan_tiles(const Plan& plan, int phase, int bm, int bn, int bk, int n_sms,
                    bool by_cost = true);

// The tile lists of a persistent launch (all phases of all iterations in one launch, each
// tile waiting until its matrix has finished the phase it reads): one list per
// q = 3 * iteration + phase for q < 3 * iters, each with `units` entries in cta_begin.
// The assignment follows a simulated run in cost units (k-blocks plus an epilogue
// allowance per tile).  A tile is ready once every tile of its matrix's previous phase
// (the previous iteration's Update, for a Gram tile) has been published: a tile is
// published kPublishLag after the next tile of its list ends, or after itself ends when
// it is the last of its list (the kernel's epilogue waits for a tile's stores at the end
// of the next one).  A phase's tiles, by readiness and then longest first, each go to
// the unit that frees first, and each unit runs its tiles in that order.  The simulation
// is causal, so the first lists do not depend on `iters`.
std::vector<TileList> plan_persistent(const Plan& plan, int bm, int bn, int bk, int units,
                                      int iters);
constexpr int64_t kPublishLag = 2;

// Owner of every matrix parameter for an n_shards-rank data-parallel group (one shard per
// rank): longest Newton-Schulz cost first, each to the least-loaded rank among those that
// hold a shard of it (ties: lowest rank).  owner[i] = -1 for non-matrix parameters;
// rank_cost[r] receives each rank's total cost in flops for ns_steps iterations.
void assign_owners(const Plan& plan, int ns_steps, int32_t* owner, double* rank_cost);

// One run of consecutive flat elements of one matrix parameter that the owner exchange
// moves between a rank's shard and the owner's packed buffer (same layout as muon_xfer).
struct XferRun {
  int32_t param;
  int32_t src_rank;   // rank (= shard index) whose shard holds the run
  int32_t dst_rank;   // the parameter's owner
  int32_t pad_;
  int64_t shard_off;  // element offset of the run in src_rank's shard
  int64_t owner_off;  // element offset of the run in dst_rank's packed buffer
  int64_t len;        // elements
};

// The owner exchange of every matrix parameter (owner[i] in 0..n_shards-1 for matrices):
// each parameter's flat range cut at shard edges into runs.  owner_offsets[i] (n_params
// entries) receives parameter i's offset in its owner's packed buffer (the parameters a
// rank owns, row-major, back to back in parameter order, each starting at a multiple of
// 4 elements), -1 for non-matrix parameters; owned_numel[r] (n_shards entries) the length
// of rank r's packed buffer.  Returns "" or a message (an owner out of range).
std::string exchange_runs(const Plan& plan, const int32_t* owner, std::vector<XferRun>* runs,
                          std::vector<int64_t>* owner_offsets, std::vector<int64_t>* owned_numel);

}  // namespace muon
