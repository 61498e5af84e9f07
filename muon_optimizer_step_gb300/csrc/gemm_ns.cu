// bf16 Newton-Schulz on the sm_103a tensor cores (tcgen05 + TMEM + TMA): the phases of
// every matrix of a flat buffer as grouped launches, one per phase, or (when pinned) all
// of them in one persistent, cooperative launch.
//
// Phases of one iteration (quintic Newton-Schulz, (a, b, c) = (3.4445, -4.7750, 2.0315)):
//   Gram    A = X X^T             (tall X: A = X^T X)      upper-triangle tiles, mirrored
//   Poly    B' = b*A + c*A A + a*I (A symmetric)           upper-triangle tiles, mirrored
//   Update  X' = s * B' X         (tall X: X' = s * X B')
// (split fp32: Poly B = b*A + c*A A, Update X' = s*(a*X + B X))
// a*X + B X = (a*I + B) X, so on the bf16 path the Poly epilogue adds a to the diagonal of
// B and the Update is a plain product: its epilogue reads no X.  (In bf16 the diagonal
// entries a + B_ii round to 8 significant bits; on the tested shapes this raises the
// update's error by 5-10 % of itself, e.g. 0.0095 to 0.0105 on 768 x 2304, within the
// 2e-2 bound.)  The split-fp32 form keeps a*X + B X: with the large diagonal inside the
// product, its full-size error rose from 6e-5 to 2e-4, over its 1e-4 bound.
// s = 1/||X||_F in the first iteration (the Gram epilogue takes s^2), 1 after it.  X keeps
// its stored row-major orientation; a tall matrix's transposes are MN-major operand reads.
// The last Update can also apply W <- W*(1 - lr*wd) - lr*sqrt(max(1, r/c))*O from the fp32 O.
//
// Scheduling: the host deals the tiles to CTAs, per phase (longest first) when each phase
// is a launch of its own.  A persistent launch walks, per CTA, one list per iteration and
// phase (Gram, Poly, Update of iteration 0, then 1, ...).  A tile starts when the phase it
// reads is complete *for its own matrix*: per matrix and phase a counter in the workspace
// counts finished CTA-tiles (release after the epilogue's stores; acquire + an async-proxy
// fence before the TMA reads).  Matrices therefore flow through the phases independently,
// and the tail of one phase overlaps the start of the next; the host orders each list by
// when its tiles' inputs are expected to be complete (a simulated run).  Every CTA's lists
// are in phase order and all CTAs are co-resident (cooperative launch, one CTA per SM):
// the lowest unfinished phase only waits on finished ones, so some CTA can always
// progress, whatever the order inside a list; every wait is bounded anyway.
//
// Three tile shapes share this code:
//   ns_tc_single_kernel: one CTA per 128 x 256 output tile, tcgen05.mma.cta_group::1, M=128 N=256;
//   ns_tc_pair_kernel: a 2-CTA cluster per 256 x 256 tile; CTA r loads rows [128r, 128r+128)
//                  of the A and of the B operand, the even CTA issues
//                  tcgen05.mma.cta_group::2 (M=256 N=256) over both CTAs' shared memory and
//                  each CTA drains its own 128 accumulator rows.  A third less operand
//                  traffic per k-block;
//   ns_tc_pairwide_kernel: a 2-CTA cluster per 256 x 512 tile: per k-step two such MMAs
//                  (N = 256 column groups 0 and 1) into one 512-column accumulator; CTA r
//                  loads its 128 rows of A and 128 rows of each group's B.  Half the
//                  operand bytes per flop of single CTAs, but the accumulator fills TMEM,
//                  so a tile's epilogue does not overlap the next tile's MMAs.
// CTA roles (384 threads): warp 0 (lane 0) issues the TMA loads, warp 1 (lane 0) the MMAs,
// warp 2 allocates TMEM, warps 4-11 drain TMEM (two warps per TMEM lane quarter warp % 4,
// half the columns each) through the epilogue.  Registers are split per SM sub-partition:
// three warps of a sub-partition share 16K registers, hence at most 168 per thread.
#include <cstdio>
#include <string>
#include <vector>

#include <cudaTypedefs.h>

#include "device_common.cuh"
#include "kernels.h"

namespace muon {

namespace {

constexpr int NUM_THREADS = 384;  // 12 warps: producer, MMA issuer, TMEM allocator, idle, 8 epilogue
constexpr int EPI_WARPS = 8;
constexpr int EPI_THREADS = EPI_WARPS * 32;
constexpr int BN = 256;             // output tile columns
constexpr int TMEM_COLS = 512;      // two 128 x 256 fp32 accumulators
constexpr float kA = 3.4445f, kB = -4.7750f, kC = 2.0315f;

// Kernel variants of one tile shape:
//   kVarTma:   bf16 operands; the epilogue stages 32 x 32 blocks in shared memory for TMA
//              bulk stores;
//   kVarSplit: the split-fp32 form: every fp32 operand kept as three bf16 parts h, m, l,
//              six kind::f16 MMAs per product (hh + hm + mh + hl + lh + mm); plain-store
//              epilogue.
// (A bf16 pair variant that traded the staging buffers for a seventh operand stage and a
// plain-store epilogue measured 3-20% slower than kVarTma: the stores cost more than the
// deeper pipeline saves.)
constexpr int kVarTma = 0, kVarSplit = 1;

template <int kShape, int kVar = kVarTma>
struct Cfg {
  static constexpr bool kSplit = kVar == kVarSplit;
  static constexpr bool kCluster = kShape != kShapeSingle;  // a 2-CTA cluster per tile
  static constexpr bool kTwoSm = kShape != kShapeSingle;    // tcgen05 cta_group::2
  static constexpr bool kWide = kShape == kShapePairWide;   // 256 x 512 tiles
  static constexpr int TILE_N = kWide ? 512 : BN;           // output tile columns
  static constexpr int ACC_BUFS = kWide ? 1 : 2;  // accumulators in TMEM's 512 columns
  static constexpr int NHALF = kWide ? 2 : 1;     // N = 256 column groups per k-step
  static constexpr int BK = 64;                       // k-block: one 128-byte row of bf16
  static constexpr int UMMA_K = 16;                   // K of one MMA: 32 bytes of a row
  static constexpr int PARTS = kSplit ? 3 : 1;        // operand copies: h (m, l)
  static constexpr int MN_W = 64;                     // MN extent of an MN-major box
  static constexpr int MN_BOX = BK * 128;             // bytes of an MN-major box (BK rows)
  static constexpr int MMA_M = kTwoSm ? 256 : 128;    // rows of one MMA instruction
  static constexpr int BROWS = kCluster ? 128 : 256;  // B-operand rows this CTA loads
  static constexpr int A_PART = 128 * 128;            // 16 KB: 128 rows of 128 bytes
  // B rows held in this CTA's stage: its own half of each N = 256 group (pairs), or all
  // 256 (single)
  static constexpr int B_PART = (kTwoSm ? 128 * NHALF : 256) * 128;
  static constexpr int A_BYTES = A_PART * PARTS;
  static constexpr int B_BYTES = B_PART * PARTS;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGING = kVar == kVarTma ? EPI_WARPS * 4096 : 0;  // 4 KB per warp
  static constexpr int STAGES = kTwoSm ? (kSplit ? 2 : (kWide ? 4 : 6)) : 4;
  static_assert(kVar == kVarTma || kTwoSm, "the plain-store variants run on CTA pairs only");
  // operand stages, epilogue staging, alignment, barriers
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + STAGING + 1024 + 256;
  static_assert(SMEM_BYTES <= 232448, "more than the 227 KB of shared memory a CTA can have");
};

struct NsParams {
  const TileDev* tiles;      // every tile list, back to back
  const int32_t* begin;      // list l, unit u: tiles [begin[l*begin_stride+u], begin[...+u+1])
  int begin_stride;          // units + 1
  int n_lists;               // 3 (one per phase) or 3 x iterations (persistent)
  const MatDev* mats;
  const CUtensorMap* tmaps;
  uint8_t* ws;
  const float* inv_norm;
  int* counters;             // per matrix and phase: finished CTA-tiles (zeroed per call)
  int* err;
  long long budget;
  int ns_steps;
  int q_begin, q_end;        // this launch runs phases q = 3*it + phase in [q_begin, q_end)
  int apply;                 // last Update also applies the step to W
  ApplyArgs ap;
  int64_t n_tiles;           // entries of `tiles`
  DebugCtx dbg;
};

// The offsets of unit `unit` in the tile list of q = 3 * it + phase (its own list, or for
// iterations past the lists the last iteration's).
__device__ __forceinline__ const int32_t* list_begin(const NsParams& p, int qq, int unit) {
  const int l = qq < p.n_lists ? qq : p.n_lists - 3 + qq % 3;
  return p.begin + (int64_t)l * p.begin_stride + unit;
}

// Debug builds: every tile this CTA (pair) will run in this launch, checked before any
// role starts.  The answer depends on the tables only, so both CTAs of a pair reach the
// same one and leave together.
template <int kShape>
__device__ __forceinline__ bool debug_tiles_ok(const NsParams& p, int unit) {
  constexpr int bm = kShape == kShapeSingle ? 128 : 256;
  if (p.n_lists < 3 || p.n_lists % 3 != 0 || unit + 1 >= p.begin_stride) return false;
  for (int qq = p.q_begin; qq < p.q_end; ++qq) {
    const int phase = qq % 3;
    const int32_t* bg = list_begin(p, qq, unit);
    const int b0 = bg[0], b1 = bg[1];
    if (b0 < 0 || b1 < b0 || b1 > p.n_tiles) return false;
    for (int ti = b0; ti < b1; ++ti) {
      const TileDev t = p.tiles[ti];
      if (!debug_tile_ok(t, phase, p.mats, p.dbg, bm, Cfg<kShape>::TILE_N, 64)) return false;
      if (p.apply && phase == kPhaseUpdate && !debug_apply_ok(p.ap, p.mats[t.mat], p.dbg))
        return false;
    }
  }
  return true;
}

// Which tensor maps and transpose bits a tile of `phase` uses.
struct TileOps {
  int a_map, b_map;
  int a_mn, b_mn;
};

template <bool kCluster>
__device__ __forceinline__ TileOps tile_ops(const MatDev& mt, int phase, int x_in) {
  const int xk = x_in ? kMapX1K128 : kMapX0K128;
  const int xkb = kCluster ? xk : (x_in ? kMapX1K256 : kMapX0K256);
  const int xmn = x_in ? kMapX1MN : kMapX0MN;
  TileOps o;
  if (phase == kPhaseGram) {
    if (mt.tall) { o.a_map = xmn; o.b_map = xmn; o.a_mn = 1; o.b_mn = 1; }
    else { o.a_map = xk; o.b_map = xkb; o.a_mn = 0; o.b_mn = 0; }
  } else if (phase == kPhasePoly) {
    o.a_map = kMapAK128; o.b_map = kCluster ? kMapAK128 : kMapAK256; o.a_mn = 0; o.b_mn = 0;
  } else {
    if (mt.tall) { o.a_map = xk; o.b_map = kCluster ? kMapBK128 : kMapBK256; o.a_mn = 0; o.b_mn = 0; }
    else { o.a_map = kMapBK128; o.b_map = xmn; o.a_mn = 0; o.b_mn = 1; }
  }
  return o;
}

// A 256-column tile whose second 128 columns lie past the matrix computes its first 128
// only (N = 128 MMAs).  On a CTA pair each CTA then holds 64 rows of B (the pair's MMA
// takes N/2 of B from each CTA), so its B rows start 64, not 128, after the tile's.
template <bool kNarrowable>
__device__ __forceinline__ bool narrow_tile(const MatDev& mt, const TileDev& tile, int phase) {
  const int n_out = phase == kPhaseUpdate ? mt.cols : mt.m;
  return kNarrowable && tile.j0 + 128 >= n_out;
}

// The counter a tile of (it, phase) waits on, and the value that means "complete".
__device__ __forceinline__ int dep_slot(const MatDev& mt, int mat, int it, int phase,
                                        int* target) {
  if (phase == kPhaseGram) {
    *target = it * mt.sig[kPhaseUpdate];
    return mat * 3 + kPhaseUpdate;
  }
  *target = (it + 1) * mt.sig[phase - 1];
  return mat * 3 + phase - 1;
}

__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Waits (bounded) until *c >= target; then orders later async-proxy (TMA) reads after the
// data the counter publishes.
__device__ __forceinline__ bool wait_counter(const int* c, int target, long long budget, int* err,
                                             volatile int* abort) {
  if (target > 0 && ld_acquire_gpu(c) < target) {
    const long long t0 = clock64();
    while (ld_acquire_gpu(c) < target) {
      if (*abort) return false;
      if (clock64() - t0 > budget) {
        atomicExch(err, kErrTimeout);
        *abort = 1;
        return false;
      }
      __nanosleep(128);
    }
  }
  asm volatile("fence.proxy.async.global;" ::: "memory");
  return true;
}

__device__ __forceinline__ void signal_counter(int* c) {
  asm volatile("fence.acq_rel.gpu;\n\tred.relaxed.gpu.global.add.s32 [%0], 1;" ::"l"(c) : "memory");
}

__device__ __forceinline__ void unpack_bf16x32(const uint4 (&u)[4], float (&f)[32]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    f[8 * q + 0] = bf16_lo(u[q].x); f[8 * q + 1] = bf16_hi(u[q].x);
    f[8 * q + 2] = bf16_lo(u[q].y); f[8 * q + 3] = bf16_hi(u[q].y);
    f[8 * q + 4] = bf16_lo(u[q].z); f[8 * q + 5] = bf16_hi(u[q].z);
    f[8 * q + 6] = bf16_lo(u[q].w); f[8 * q + 7] = bf16_hi(u[q].w);
  }
}

// The global input an epilogue chunk needs besides the accumulator (A, for Poly only),
// loaded one chunk ahead so that its memory latency overlaps the previous chunk.
// Returns false when the chunk needs none or takes the element-by-element path.
__device__ __forceinline__ bool epilogue_prefetch(const NsParams& p, const MatDev& mt, int phase,
                                                  int i, int jb, uint4 (&in)[4]) {
  const uint4* src;
  if (phase == kPhasePoly) {
    if (i >= mt.m || jb + 32 > mt.m || jb + 31 < i) return false;
    src = reinterpret_cast<const uint4*>(p.ws + mt.a + 2 * ((int64_t)i * mt.lda + jb));
  } else {
    return false;
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) in[q] = src[q];
  return true;
}

// Per-warp staging of one 32 x 32 output block (and its transposed mirror) in shared
// memory, laid out as the 64-byte-swizzled boxes the TMA stores read: element (row r,
// column c) of a block sits at byte 64 r + 16 ((c / 8) ^ ((r / 2) % 4)) + 2 (c % 8).
struct EpiStage {
  uint8_t* dir;   // 2 KB, 512-byte aligned
  uint8_t* mir;   // 2 KB
  bool pending;   // a bulk store may still be reading these buffers (tracked by lane 0)
  int groups;     // bulk-store groups committed for the current tile
};

__device__ __forceinline__ uint32_t swz64(int r, int c) {
  return (uint32_t)(64 * r + 16 * ((c >> 3) ^ ((r >> 1) & 3)) + 2 * (c & 7));
}

// Epilogue of the 32 x 32 block: rows r0 .. r0+31 (lane = row - r0), accumulator columns
// [jb, jb+32).  `in` holds the prefetched A row segment (Poly) when have_in.  Full blocks
// leave through TMA bulk stores (direct block, and its mirror for the symmetric outputs);
// blocks on the diagonal of a symmetric output keep the element rule (j >= i written,
// j > i mirrored) so that every element has exactly one writer.
__device__ __forceinline__ void epilogue_block(const NsParams& p, const MatDev& mt, int mat,
                                               int phase, int x_in, bool apply, int r0, int jb,
                                               int lane, const uint32_t (&acc)[32], float s,
                                               const uint4 (&in)[4], bool have_in,
                                               EpiStage& st) {
  const int i = r0 + lane;
  float f[32];
  const CUtensorMap* maps = p.tmaps + (size_t)mat * kMapsPerMat;
  const CUtensorMap* out_map;
  bool mirror = false;
  if (phase == kPhaseUpdate) {
    if (r0 >= mt.rows || jb >= mt.cols) return;  // warp-uniform
#pragma unroll
    for (int t = 0; t < 32; ++t) f[t] = s * __uint_as_float(acc[t]);
    if (apply) {
      // The staging buffers (4 KB) turn the block around for coalesced weight accesses,
      // once the previous bulk store has read them.
      if (st.pending) {
        if (lane == 0) bulk_wait_read();
        __syncwarp();
      }
      apply_block(p.ap, mt, r0, jb, lane, f, st.dir);
    }
    out_map = maps + (x_in ? kMapX0St : kMapX1St);
  } else {
    if (r0 >= mt.m || jb >= mt.m || jb < r0) return;  // outside, or below the diagonal
    __nv_bfloat16* am = reinterpret_cast<__nv_bfloat16*>(p.ws + mt.a);
    const int64_t row = (int64_t)i * mt.lda;
    if (phase == kPhaseGram) {
#pragma unroll
      for (int t = 0; t < 32; ++t) f[t] = __uint_as_float(acc[t]) * s;
    } else {
      float a[32];
      if (have_in) {
        unpack_bf16x32(in, a);
      } else {
#pragma unroll
        for (int t = 0; t < 32; ++t)
          a[t] = (i < mt.m && jb + t < mt.m) ? __bfloat162float(am[row + jb + t]) : 0.f;
      }
#pragma unroll
      for (int t = 0; t < 32; ++t) f[t] = fmaf(kB, a[t], kC * __uint_as_float(acc[t]));
    }
    if (jb == r0) {
      // Diagonal block: element rule with plain stores; Poly adds a on the diagonal.
      __nv_bfloat16* out = phase == kPhaseGram ? am : reinterpret_cast<__nv_bfloat16*>(p.ws + mt.b);
      const float diag = phase == kPhasePoly ? kA : 0.f;
      if (i < mt.m) {
#pragma unroll
        for (int t = 0; t < 32; ++t) {
          const int j = jb + t;
          if (j >= i && j < mt.m) out[row + j] = __float2bfloat16_rn(j == i ? f[t] + diag : f[t]);
          if (j > i && j < mt.m) out[(int64_t)j * mt.lda + i] = __float2bfloat16_rn(f[t]);
        }
      }
      return;
    }
    out_map = maps + (phase == kPhaseGram ? kMapASt : kMapBSt);
    mirror = true;
  }
  // Full block through shared memory and TMA (out-of-range rows / columns are clipped by
  // the tensor map, so their values do not matter).
  if (st.pending) {
    if (lane == 0) bulk_wait_read();
    __syncwarp();
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint4 u;
    u.x = pack_bf16x2(f[8 * k + 0], f[8 * k + 1]);
    u.y = pack_bf16x2(f[8 * k + 2], f[8 * k + 3]);
    u.z = pack_bf16x2(f[8 * k + 4], f[8 * k + 5]);
    u.w = pack_bf16x2(f[8 * k + 6], f[8 * k + 7]);
    *reinterpret_cast<uint4*>(st.dir + swz64(lane, 8 * k)) = u;
  }
  if (mirror) {
#pragma unroll
    for (int t = 0; t < 32; ++t)
      *reinterpret_cast<__nv_bfloat16*>(st.mir + swz64(t, lane)) = __float2bfloat16_rn(f[t]);
  }
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    // Outputs are read again only by the next phase: store them evict-first, so that
    // they do not push out the operand panels this phase's tiles are still streaming.
    const uint64_t pol = l2_policy_evict_first();
    tma_store_2d_hint(out_map, jb, r0, smem_u32(st.dir), pol);
    if (mirror) tma_store_2d_hint(out_map, r0, jb, smem_u32(st.mir), pol);
    bulk_commit();
  }
  st.pending = true;
  ++st.groups;
}

// ---------------------------------------------------------------- plain-store epilogue
// Values kept as P bf16 parts in P equal arrays, `part` elements apart: P = 1 is plain
// bf16, P = 3 the split-fp32 form (h, m, l).
template <int P>
__device__ __forceinline__ void split_parts(float x, __nv_bfloat16 (&q)[P]) {
  if constexpr (P == 1) q[0] = __float2bfloat16_rn(x);
  else split_bf16x3(x, q[0], q[1], q[2]);
}

// Row run of 32 values at element index e: loads the sum of the parts, or stores the
// parts of f.  n < 32 takes the first n only.
template <int P>
__device__ __forceinline__ void load_split_run(const __nv_bfloat16* h, int64_t part, int64_t e,
                                               int n, float (&x)[32]) {
  if (n == 32) {
#pragma unroll
    for (int t = 0; t < 32; ++t) x[t] = 0.f;
#pragma unroll
    for (int k = P - 1; k >= 0; --k) {  // smallest part first
      uint4 u[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) u[q] = *reinterpret_cast<const uint4*>(h + k * part + e + 8 * q);
      float v[32];
      unpack_bf16x32(u, v);
#pragma unroll
      for (int t = 0; t < 32; ++t) x[t] = v[t] + x[t];
    }
  } else {
#pragma unroll
    for (int t = 0; t < 32; ++t) {
      float v = 0.f;
#pragma unroll
      for (int k = P - 1; k >= 0; --k) v = (t < n ? __bfloat162float(h[k * part + e + t]) : 0.f) + v;
      x[t] = v;
    }
  }
}

template <int P>
__device__ __forceinline__ void store_split1(__nv_bfloat16* h, int64_t part, int64_t e, float f) {
  __nv_bfloat16 q[P];
  split_parts<P>(f, q);
#pragma unroll
  for (int k = 0; k < P; ++k) h[k * part + e] = q[k];
}

template <int P>
__device__ __forceinline__ void store_split_run(__nv_bfloat16* h, int64_t part, int64_t e, int n,
                                                const float (&f)[32]) {
  if (n == 32) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t w[P][4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        __nv_bfloat16 a[P], b[P];
        split_parts<P>(f[8 * q + 2 * k], a);
        split_parts<P>(f[8 * q + 2 * k + 1], b);
#pragma unroll
        for (int c = 0; c < P; ++c)
          w[c][k] = (uint32_t)__bfloat16_as_ushort(a[c]) | ((uint32_t)__bfloat16_as_ushort(b[c]) << 16);
      }
#pragma unroll
      for (int c = 0; c < P; ++c)
        *reinterpret_cast<uint4*>(h + c * part + e + 8 * q) = make_uint4(w[c][0], w[c][1], w[c][2], w[c][3]);
    }
  } else {
#pragma unroll
    for (int t = 0; t < 32; ++t)
      if (t < n) store_split1<P>(h, part, e + t, f[t]);
  }
}

// Epilogue of a 32 x 32 block with plain stores: the same arithmetic as epilogue_block
// on fp32 values (inputs: the sum of the P parts), written back as P bf16 parts: the row
// run of each lane, and for symmetric outputs the transposed block, whose stores are
// coalesced across the warp (lane = column of the mirror row).  Diagonal blocks keep the
// element rule (j >= i written, j > i mirrored).  It needs no shared memory, which leaves
// room for the split form's wider stages.
template <int P>
__device__ __forceinline__ void epilogue_block_plain(const NsParams& p, const MatDev& mt,
                                                     int phase, int x_in, bool apply, int r0,
                                                     int jb, int lane, const uint32_t (&acc)[32],
                                                     float s) {
  const int i = r0 + lane;
  float f[32];
  if (phase == kPhaseUpdate) {
    if (r0 >= mt.rows || jb >= mt.cols) return;  // warp-uniform
    const int64_t part = split_part_bytes((int64_t)mt.rows * mt.ldx * 2) / 2;
    const __nv_bfloat16* xin = reinterpret_cast<const __nv_bfloat16*>(p.ws + (x_in ? mt.x1 : mt.x0));
    __nv_bfloat16* xout = reinterpret_cast<__nv_bfloat16*>(p.ws + (x_in ? mt.x0 : mt.x1));
    const int n = i < mt.rows ? min(32, mt.cols - jb) : 0;
    const int64_t e = (int64_t)i * mt.ldx + jb;
    float x[32];
    load_split_run<P>(xin, part, e, n, x);
#pragma unroll
    for (int t = 0; t < 32; ++t) f[t] = s * fmaf(kA, x[t], __uint_as_float(acc[t]));
    if (apply && n > 0) apply_row_run(p.ap, mt, i, jb, n, f);
    if (n > 0) store_split_run<P>(xout, part, e, n, f);
    return;
  }
  if (r0 >= mt.m || jb >= mt.m || jb < r0) return;  // outside, or below the diagonal
  const int64_t part = split_part_bytes((int64_t)mt.m * mt.lda * 2) / 2;
  __nv_bfloat16* am = reinterpret_cast<__nv_bfloat16*>(p.ws + mt.a);
  const int n = i < mt.m ? min(32, mt.m - jb) : 0;
  const int64_t e = (int64_t)i * mt.lda + jb;
  if (phase == kPhaseGram) {
#pragma unroll
    for (int t = 0; t < 32; ++t) f[t] = __uint_as_float(acc[t]) * s;
  } else {
    float a[32];
    load_split_run<P>(am, part, e, n, a);
#pragma unroll
    for (int t = 0; t < 32; ++t) f[t] = fmaf(kB, a[t], kC * __uint_as_float(acc[t]));
  }
  __nv_bfloat16* out = phase == kPhaseGram ? am : reinterpret_cast<__nv_bfloat16*>(p.ws + mt.b);
  if (jb == r0) {
    if (i < mt.m) {
#pragma unroll
      for (int t = 0; t < 32; ++t) {
        const int j = jb + t;
        if (j >= i && j < mt.m) store_split1<P>(out, part, (int64_t)i * mt.lda + j, f[t]);
        if (j > i && j < mt.m) store_split1<P>(out, part, (int64_t)j * mt.lda + i, f[t]);
      }
    }
    return;
  }
  if (n > 0) store_split_run<P>(out, part, e, n, f);
  if (i < mt.m) {
#pragma unroll
    for (int t = 0; t < 32; ++t)
      if (jb + t < mt.m) store_split1<P>(out, part, (int64_t)(jb + t) * mt.lda + i, f[t]);
  }
}

// Bounded wait; on expiry also tells the peer CTA of a pair to stop.
template <bool kCluster>
__device__ __forceinline__ bool wait_role(uint64_t* bar, uint32_t parity, const NsParams& p,
                                          volatile int* abort, uint32_t peer_abort) {
  if (mbar_wait_bounded(bar, parity, p.budget, p.err, abort)) return true;
  if (kCluster) asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(peer_abort), "r"(1) : "memory");
  return false;
}

// Bounded wait that ignores the abort flag: drains copies and MMAs already in flight.
__device__ __forceinline__ bool wait_drain(uint64_t* bar, uint32_t parity, long long budget,
                                           int* err) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > budget) {
      atomicExch(err, kErrTimeout);
      return false;
    }
  }
  return true;
}

// Epilogue threads agree on stopping (any thread saw an abort or a failed wait).
__device__ __forceinline__ bool epi_any(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "n"(EPI_THREADS)
      : "memory");
  return r != 0;
}

template <int kShape, int kVar = kVarTma>
__device__ __forceinline__ void ns_tc_body(const NsParams& p) {
  using C = Cfg<kShape, kVar>;
  constexpr bool kSplit = C::kSplit;
  constexpr bool kCluster = C::kCluster;
  constexpr bool kTwoSm = C::kTwoSm;
  extern __shared__ uint8_t smem_raw[];
  __shared__ int abort_flag;
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* tiles_smem = smem_raw + pad;
  uint64_t* bars = reinterpret_cast<uint64_t*>(tiles_smem + C::STAGES * C::STAGE_BYTES +
                                               C::STAGING);
  uint64_t* full = bars;
  uint64_t* empty = bars + C::STAGES;
  uint64_t* acc_full = bars + 2 * C::STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* mma_done = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = kCluster ? cluster_ctarank() : 0u;  // pair: 0 issues the MMAs
  const int unit = kCluster ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  if constexpr (kDebugChecks) {
    __shared__ int dbg_bad;
    if (threadIdx.x == 0) {
      dbg_bad = debug_tiles_ok<kShape>(p, unit) ? 0 : 1;
      if (dbg_bad) debug_fail(p.dbg);
    }
    __syncthreads();
    if (dbg_bad) return;
  }
  const uint32_t peer_abort = kCluster ? mapa_shared(smem_u32(&abort_flag), rank ^ 1u) : 0u;
  // This CTA issues MMAs (all but the odd CTA of a cta_group::2 pair).
  const bool mma_cta = !kTwoSm || rank == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);   // the (pair: even) CTA's arrival with the expected bytes
      mbar_init(&empty[s], 1);  // the MMA commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], (kTwoSm ? 2 : 1) * EPI_WARPS);
    }
    mbar_init(mma_done, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 2) {
    if (kTwoSm) {
      tmem_alloc_pair(tmem_slot, TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_slot, TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  if (kCluster) cluster_sync(); else __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  volatile int* abort = &abort_flag;
  // Several phases in this launch: tiles wait on, and publish to, the per-matrix counters.
  const bool chained = p.q_end - p.q_begin > 1;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t ph = 0;
      long long nfill = 0;
      bool ok = true;
      for (int qq = p.q_begin; qq < p.q_end && ok; ++qq) {
        const int it = qq / 3, phase = qq % 3;
        {
          const int x_in = it & 1;
          const int32_t* bg = list_begin(p, qq, unit);
          for (int ti = bg[0]; ti < bg[1] && ok; ++ti) {
            const TileDev tile = p.tiles[ti];
            const MatDev& mt = p.mats[tile.mat];
            int target;
            const int slot = dep_slot(mt, tile.mat, it, phase, &target);
            // One phase per launch: stream order already made the inputs complete.
            if (!chained) target = 0;
            if (!wait_counter(p.counters + slot, target, p.budget, p.err, abort)) {
              if (kCluster)
                asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(peer_abort), "r"(1) : "memory");
              ok = false;
              break;
            }
            const TileOps ops = tile_ops<kCluster>(mt, phase, x_in);
            const CUtensorMap* amap = p.tmaps + (size_t)tile.mat * kMapsPerMat + ops.a_map;
            const CUtensorMap* bmap = p.tmaps + (size_t)tile.mat * kMapsPerMat + ops.b_map;
            const int ia = tile.i0 + (kCluster ? 128 * (int)rank : 0);
            const bool narrow = narrow_tile<!C::kWide>(mt, tile, phase);
            const int jr = tile.j0 + (kCluster ? (narrow ? 64 : 128) * (int)rank : 0);
            for (int kb = 0; kb < tile.kblocks; ++kb) {
              if (!wait_role<kCluster>(&empty[stage], ph ^ 1u, p, abort, peer_abort)) {
                ok = false;
                break;
              }
              uint8_t* sa = tiles_smem + stage * C::STAGE_BYTES;
              uint8_t* sb = sa + C::A_BYTES;
              const int k0 = kb * C::BK;
              if (kTwoSm) {
                // Only the even CTA arrives, announcing both CTAs' bytes; the odd CTA's
                // copies may land first (the transaction count dips below zero, which
                // mbarriers allow; the phase still needs the even CTA's arrival).
                if (rank == 0) mbar_arrive_expect_tx(&full[stage], 2 * C::STAGE_BYTES);
                const uint32_t fbar = mapa_shared(smem_u32(&full[stage]), 0);
#pragma unroll
                for (int part = 0; part < C::PARTS; ++part) {  // h (then m, l: split fp32)
                  const CUtensorMap* am = amap + part * kMapPart;
                  const CUtensorMap* bm = bmap + part * kMapPart;
                  const uint32_t da = smem_u32(sa) + part * C::A_PART;
                  const uint32_t db = smem_u32(sb) + part * C::B_PART;
                  if (ops.a_mn) {
#pragma unroll
                    for (int q = 0; q < 128 / C::MN_W; ++q)
                      tma_load_2d_pair(da + q * C::MN_BOX, am, ia + q * C::MN_W, k0, fbar);
                  } else {
                    tma_load_2d_pair(da, am, k0, ia, fbar);
                  }
#pragma unroll
                  for (int h = 0; h < C::NHALF; ++h) {  // this CTA's 128 rows of each N group
                    const uint32_t dbh = db + h * (C::B_PART / C::NHALF);
                    const int jrh = jr + 256 * h;
                    if (ops.b_mn) {
#pragma unroll
                      for (int q = 0; q < 128 / C::MN_W; ++q)
                        tma_load_2d_pair(dbh + q * C::MN_BOX, bm, jrh + q * C::MN_W, k0, fbar);
                    } else {
                      tma_load_2d_pair(dbh, bm, k0, jrh, fbar);
                    }
                  }
                }
              } else {
                mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
                if (ops.a_mn) {
                  tma_load_2d(sa, amap, ia, k0, &full[stage]);
                  tma_load_2d(sa + C::MN_BOX, amap, ia + C::MN_W, k0, &full[stage]);
                } else {
                  tma_load_2d(sa, amap, k0, ia, &full[stage]);
                }
                if (ops.b_mn) {
#pragma unroll
                  for (int q = 0; q < C::BROWS / C::MN_W; ++q)
                    tma_load_2d(sb + q * C::MN_BOX, bmap, jr + C::MN_W * q, k0, &full[stage]);
                } else {
                  tma_load_2d(sb, bmap, k0, jr, &full[stage]);
                }
              }
              ++nfill;
              if (++stage == C::STAGES) {
                stage = 0;
                ph ^= 1u;
              }
            }
          }
        }
      }
      // Every copy issued must land before the block exits (already true unless aborted).
      // For a pair the even CTA's full barriers count both CTAs' copies.
      if (mma_cta)
        for (long long k = nfill - 1; k >= 0 && k >= nfill - C::STAGES; --k)
          wait_drain(&full[k % C::STAGES], (uint32_t)((k / C::STAGES) & 1), p.budget, p.err);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0 && mma_cta) {
      int stage = 0;
      uint32_t ph = 0;
      int lt = 0;
      bool ok = true;
      const uint32_t sbase = smem_u32(tiles_smem);
      for (int qq = p.q_begin; qq < p.q_end && ok; ++qq) {
        const int it = qq / 3, phase = qq % 3;
        {
          const int32_t* bg = list_begin(p, qq, unit);
          for (int ti = bg[0]; ti < bg[1]; ++ti, ++lt) {
            const TileDev tile = p.tiles[ti];
            const MatDev& mt = p.mats[tile.mat];
            const TileOps ops = tile_ops<kCluster>(mt, phase, it & 1);
            // Columns the epilogue would discard are not computed:
            //  - symmetric phases, single CTAs: a tile whose rows all lie at or below its
            //    second column half (i0 = j0 + 128) skips the first half (a pair's MMA
            //    covers both CTAs' rows, so it cannot skip per CTA);
            //  - a 256-column tile whose second column half lies outside the matrix skips
            //    that half (narrow_tile; on a pair the producer has placed each CTA's 64
            //    rows of the first half).
            // A half is done as N = 128 MMAs on that half of B, into that half of the
            // accumulator.
            const int row0 = tile.i0 + (kCluster ? 128 * (int)rank : 0);
            const int n_out = phase == kPhaseUpdate ? mt.cols : mt.m;
            const int m_out = phase == kPhaseUpdate ? mt.rows : mt.m;
            const bool skip_first = !kTwoSm && phase != kPhaseUpdate && tile.j0 + 128 <= row0;
            const bool skip_second = narrow_tile<!C::kWide>(mt, tile, phase);
            const bool idle = !kTwoSm && (row0 >= m_out || (skip_first && skip_second));
            const bool half_n = !idle && (skip_first || skip_second);
            const uint32_t idesc = idesc_bf16(C::MMA_M, half_n ? BN / 2 : BN, ops.a_mn, ops.b_mn);
            // 256 x 512 tiles: an N = 256 column group whose outputs the epilogue discards
            // (all left of the tile's first row in a symmetric phase, or past the matrix)
            // gets no MMAs.  The decision holds for both CTAs' rows.
            bool grp_on[C::NHALF];
#pragma unroll
            for (int h = 0; h < C::NHALF; ++h) {
              const int c0 = tile.j0 + 256 * h;
              grp_on[h] = !C::kWide ||
                          !(c0 >= n_out || (phase != kPhaseUpdate && c0 + 255 < tile.i0));
            }
            const int ab = lt % C::ACC_BUFS;
            const uint32_t use = (uint32_t)(lt / C::ACC_BUFS);
            if (!wait_role<kCluster>(&acc_empty[ab], (use & 1u) ^ 1u, p, abort, peer_abort)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t d = tmem_base + (uint32_t)(ab * BN) + (skip_first ? (uint32_t)(BN / 2) : 0u);
            for (int kb = 0; kb < tile.kblocks && ok; ++kb) {
              if (!wait_role<kCluster>(&full[stage], ph, p, abort, peer_abort)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint32_t sa = sbase + stage * C::STAGE_BYTES;
              // (the second half of B: rows 128-255 K-major, or MN-major boxes 2 and 3)
              const uint32_t sb = sa + C::A_BYTES + (skip_first ? (uint32_t)(C::B_PART / 2) : 0u);
              // One MMA reads 32 bytes of every operand row: +32 B along a K-major row, or
              // UMMA_K rows of 128 B of an MN-major box.
              constexpr uint32_t kMnStep = C::UMMA_K * 128;
#pragma unroll
              for (int kk = 0; kk < C::BK / C::UMMA_K; ++kk) {
                if (idle) break;
                const uint32_t koff_a = ops.a_mn ? kk * kMnStep : kk * 32;
                const uint32_t koff_b = ops.b_mn ? kk * kMnStep : kk * 32;
                const uint32_t lbo_a = ops.a_mn ? C::MN_BOX : 16;
                const uint32_t lbo_b = ops.b_mn ? C::MN_BOX : 16;
                const uint64_t ad = smem_desc_sw128(sa + koff_a, lbo_a, 1024);
                const uint64_t bd = smem_desc_sw128(sb + koff_b, lbo_b, 1024);
                const uint32_t acc = (kb | kk) != 0 ? 1u : 0u;
                if (kSplit) {
                  // x*y ~ hh + hm + mh + hl + lh + mm, all accumulated in fp32
                  const uint64_t ad_m = smem_desc_sw128(sa + C::A_PART + koff_a, lbo_a, 1024);
                  const uint64_t bd_m = smem_desc_sw128(sb + C::B_PART + koff_b, lbo_b, 1024);
                  const uint64_t ad_l = smem_desc_sw128(sa + 2 * C::A_PART + koff_a, lbo_a, 1024);
                  const uint64_t bd_l = smem_desc_sw128(sb + 2 * C::B_PART + koff_b, lbo_b, 1024);
                  tc_mma_f16_pair(d, ad, bd, idesc, acc);
                  tc_mma_f16_pair(d, ad, bd_m, idesc, 1u);
                  tc_mma_f16_pair(d, ad_m, bd, idesc, 1u);
                  tc_mma_f16_pair(d, ad, bd_l, idesc, 1u);
                  tc_mma_f16_pair(d, ad_l, bd, idesc, 1u);
                  tc_mma_f16_pair(d, ad_m, bd_m, idesc, 1u);
                } else if (kTwoSm) {
#pragma unroll
                  for (int h = 0; h < C::NHALF; ++h) {  // each N = 256 group of a 512-wide tile
                    if (!grp_on[h]) continue;
                    const uint64_t bdh = h == 0 ? bd
                        : smem_desc_sw128(sb + h * (C::B_PART / C::NHALF) + koff_b, lbo_b, 1024);
                    tc_mma_f16_pair(d + 256u * h, ad, bdh, idesc, acc);
                  }
                } else {
                  tc_mma_f16(d, ad, bd, idesc, acc);
                }
              }
              if (kTwoSm) tc_commit_pair(&empty[stage], (uint16_t)0x3);
              else tc_commit(&empty[stage]);
              if (++stage == C::STAGES) {
                stage = 0;
                ph ^= 1u;
              }
            }
            if (!ok) break;
            if (kTwoSm) tc_commit_pair(&acc_full[ab], (uint16_t)0x3);
            else tc_commit(&acc_full[ab]);
          }
        }
      }
      // Every MMA issued must complete before TMEM is released.
      if (kTwoSm) tc_commit_pair(mma_done, (uint16_t)0x1);
      else tc_commit(mma_done);
      wait_drain(mma_done, 0, p.budget, p.err);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- epilogue
    // Two warps per TMEM lane quarter (warp % 4), each draining half the columns.
    const int q = warp & 3;
    const int half = (warp - 4) >> 2;
    int lt = 0;
    bool stop = false;
    EpiStage est;
    est.dir = tiles_smem + C::STAGES * C::STAGE_BYTES + (warp - 4) * 4096;
    est.mir = est.dir + 2048;
    est.pending = false;
    est.groups = 0;
    int prev_slot = -1;  // counter of the previous tile, not yet published
    for (int qq = p.q_begin; qq < p.q_end && !stop; ++qq) {
      const int it = qq / 3, phase = qq % 3;
      {
        const int x_in = it & 1;
        const bool apply = p.apply && phase == kPhaseUpdate && it == p.ns_steps - 1;
        const int32_t* bg = list_begin(p, qq, unit);
        for (int ti = bg[0]; ti < bg[1]; ++ti, ++lt) {
          const TileDev tile = p.tiles[ti];
          const MatDev& mt = p.mats[tile.mat];
          const int ab = lt % C::ACC_BUFS;
          const uint32_t use = (uint32_t)(lt / C::ACC_BUFS);
          // Applying Update: while this tile's MMAs run, each lane asks L2 for the weights
          // of its row and this warp's columns, so that the epilogue's loads hit L2.
          if (apply)
            prefetch_w_row(p.ap, mt, tile.i0 + (kCluster ? 128 * (int)rank : 0) + 32 * q + lane,
                           tile.j0 + half * (C::TILE_N / 2), C::TILE_N / 2);
          bool ok = *abort == 0 && mbar_wait_bounded(&acc_full[ab], use & 1u, p.budget, p.err,
                                                     abort);
          ok = __all_sync(0xffffffffu, ok);
          if (ok) {
            tc_fence_after();
            // The epilogue reads what the previous phase wrote (A, X): acquire its counter.
            int target;
            const int slot = dep_slot(mt, tile.mat, it, phase, &target);
            if (chained && target > 0) (void)ld_acquire_gpu(p.counters + slot);
            float s = 1.f;
            if (it == 0 && phase != kPhasePoly) {
              const float inv = p.inv_norm[tile.mat];
              s = phase == kPhaseGram ? inv * inv : inv;
            }
            const int r0 = tile.i0 + (kCluster ? 128 * (int)rank : 0) + 32 * q;
            const int i = r0 + lane;
            // this warp's 32-column blocks: half of the tile's columns
            const int c_first = half * (C::TILE_N / 64), c_last = (half + 1) * (C::TILE_N / 64);
            // The X (Update) or A (Poly) input of the next 32 x 32 block is loaded before
            // this block's TMEM load and math, so that its memory latency overlaps them.
            uint4 in_next[4];
            bool have_next = false;
            if constexpr (kVar == kVarTma)
              have_next = epilogue_prefetch(p, mt, phase, i, tile.j0 + 32 * c_first, in_next);
#pragma unroll 1
            for (int c = c_first; c < c_last; ++c) {
              uint32_t v[32];
              if constexpr (kVar != kVarTma) {
                tmem_ld_32x32b_x32(
                    tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(ab * BN + 32 * c), v);
                tmem_ld_wait();
                epilogue_block_plain<C::PARTS>(p, mt, phase, x_in, apply, r0, tile.j0 + 32 * c,
                                               lane, v, s);
              } else {
                uint4 in_cur[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) in_cur[k] = in_next[k];
                const bool have_cur = have_next;
                if (c + 1 < c_last)
                  have_next = epilogue_prefetch(p, mt, phase, i, tile.j0 + 32 * (c + 1), in_next);
                tmem_ld_32x32b_x32(
                    tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(ab * BN + 32 * c), v);
                tmem_ld_wait();
                epilogue_block(p, mt, tile.mat, phase, x_in, apply, r0, tile.j0 + 32 * c, lane,
                               v, s, in_cur, have_cur, est);
              }
            }
          }
          tc_fence_before();
          __syncwarp();
          if (ok && lane == 0) {
            if (!kTwoSm || rank == 0) mbar_arrive(&acc_empty[ab]);
            else mbar_arrive_cluster(mapa_shared(smem_u32(&acc_empty[ab]), 0));
          }
          if (chained) {
            // A tile is published (its counter raised) once its bulk stores have landed.
            // Inside a list that is done at the end of the next tile, whose own stores
            // stay in flight meanwhile; the last tile of a list is published at once,
            // since a later list of this CTA may wait on it.  Tiles of one list never
            // wait on each other.
            const bool last = ti + 1 >= bg[1];
            if (last || prev_slot >= 0) {
              if (est.pending) {
                if (lane == 0) {
                  if (last) bulk_wait_all();
                  else bulk_wait_all_but(est.groups);
                  asm volatile("fence.proxy.async.global;" ::: "memory");
                }
                __syncwarp();
                est.pending = !last;
              }
              // All epilogue warps stop together, or publish together.  (Whether a tile
              // publishes depends on its place in the list only: every warp agrees.)
              stop = epi_any(!ok || *abort != 0);
              if (stop) break;
              if (warp == 4 && lane == 0) {
                if (prev_slot >= 0) signal_counter(p.counters + prev_slot);
                if (last) signal_counter(p.counters + tile.mat * 3 + phase);
              }
            }
            prev_slot = last ? -1 : tile.mat * 3 + phase;
            est.groups = 0;
          } else if (!ok) {
            stop = true;
            break;
          }
        }
      }
    }
    if (stop && kCluster)
      asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(peer_abort), "r"(1) : "memory");
    // Shared memory must outlive every bulk store that reads it.
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }
  tc_fence_before();
  if (kCluster) cluster_sync(); else __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    if (kTwoSm) tmem_dealloc_pair(tmem_base, TMEM_COLS);
    else tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// The tile shapes as separate kernels: the cluster kernels carry their cluster shape in
// their attributes, so they can be neither launched nor sized (occupancy) without it.
__global__ void __launch_bounds__(NUM_THREADS, 1)
    ns_tc_single_kernel(const __grid_constant__ NsParams p) {
  ns_tc_body<kShapeSingle>(p);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
    ns_tc_pair_kernel(const __grid_constant__ NsParams p) {
  ns_tc_body<kShapePair>(p);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
    ns_tc_pairwide_kernel(const __grid_constant__ NsParams p) {
  ns_tc_body<kShapePairWide>(p);
}

// The split-fp32 form, on CTA pairs.
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
    ns_tc_split_kernel(const __grid_constant__ NsParams p) {
  ns_tc_body<kShapePair, kVarSplit>(p);
}

using NsKernel = void (*)(NsParams);

template <int kShape>
NsKernel ns_tc_kernel_of() {
  return kShape == kShapeSingle ? ns_tc_single_kernel
         : kShape == kShapePair ? ns_tc_pair_kernel : ns_tc_pairwide_kernel;
}

__global__ void selftest_timeout_kernel(int* err, long long budget) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // Nobody arrives on `bar`: the wait must run out, record the timeout and return.
  if (threadIdx.x == 0) mbar_wait_bounded(&bar, 0, budget, err, &abort_flag);
}

template <int kShape, int kVar = kVarTma>
cudaError_t launch_impl(const Plan& plan, const DevTables& dt, void* ws, int ns_steps,
                        int q_begin, int q_end, long long budget, const ApplyArgs* ap,
                        cudaStream_t st) {
  uint8_t* w = static_cast<uint8_t*>(ws);
  NsParams p;
  p.tiles = dt.tc_tiles;
  p.begin = dt.tc_begin;
  p.begin_stride = dt.tc_units + 1;
  p.n_lists = dt.tc_lists;
  p.mats = dt.mats;
  p.tmaps = dt.tmaps;
  p.ws = w;
  p.inv_norm = reinterpret_cast<const float*>(w + plan.ws_inv_norm);
  p.counters = reinterpret_cast<int*>(w + plan.ws_counters);
  p.err = dt.err;
  p.budget = budget;
  p.ns_steps = ns_steps;
  p.q_begin = q_begin;
  p.q_end = q_end;
  p.apply = ap != nullptr ? 1 : 0;
  if (ap != nullptr) p.ap = *ap;
  p.n_tiles = dt.tc_n_tiles;
  p.dbg = make_debug_ctx(plan, dt);
  cudaError_t e = cudaSuccess;
  if (q_end - q_begin > 1) {
    e = cudaMemsetAsync(p.counters, 0, plan.mats.size() * 3 * sizeof(int), st);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  constexpr bool kCluster = Cfg<kShape, kVar>::kCluster;
  const NsKernel kernel = kVar == kVarSplit ? ns_tc_split_kernel : ns_tc_kernel_of<kShape>();
  cfg.gridDim = dim3((unsigned)((kCluster ? 2 : 1) * dt.tc_units), 1, 1);
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = Cfg<kShape, kVar>::SMEM_BYTES;
  cfg.stream = st;
  // A persistent launch (several phases) needs every CTA resident at once, because tiles
  // wait on tiles of other CTAs.  Single CTAs ask for a cooperative launch.  Cluster
  // kernels are launched without that attribute, with a grid sized to the device's
  // resident-cluster count (occupancy query), so that no launch can fail and be retried
  // (which would also break stream capture).  One phase per launch needs neither.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = (q_end - q_begin > 1 && !kCluster) ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, kernel, p);
  return e;
}

}  // namespace

cudaError_t prepare_ns_kernels(int* max_pairs, int* max_singles) {
  const void* fns[4] = {(const void*)ns_tc_single_kernel, (const void*)ns_tc_pair_kernel,
                        (const void*)ns_tc_split_kernel, (const void*)ns_tc_pairwide_kernel};
  const int smems[4] = {Cfg<kShapeSingle>::SMEM_BYTES, Cfg<kShapePair>::SMEM_BYTES,
                        Cfg<kShapePair, kVarSplit>::SMEM_BYTES,
                        Cfg<kShapePairWide>::SMEM_BYTES};
  for (int k = 0; k < 4; ++k) {
    const void* fn = fns[k];
    const int smem = smems[k];
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
  }
  int per_sm = 0, sms = 0, dev = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      &per_sm, ns_tc_single_kernel, NUM_THREADS, Cfg<kShapeSingle>::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  *max_singles = per_sm * sms;
  // Resident 2-CTA clusters: the smallest count of the cluster kernels.
  int n_min = 1 << 30;
  for (int k = 1; k < 4; ++k) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * 1024, 1, 1);
    cfg.blockDim = dim3(NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = smems[k];
    int n = 0;
    const NsKernel kern = k == 1 ? ns_tc_pair_kernel
                          : k == 2 ? ns_tc_split_kernel : ns_tc_pairwide_kernel;
    e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    if (e != cudaSuccess) return e;
    n_min = n < n_min ? n : n_min;
  }
  *max_pairs = n_min;
  return cudaSuccess;
}

cudaError_t launch_ns_tc(const Plan& plan, const DevTables& dt, void* ws, int ns_steps,
                         long long budget, const ApplyArgs* ap, cudaStream_t st) {
  if (dt.tc_units == 0 || ns_steps == 0) return cudaSuccess;
  const int nq = 3 * ns_steps;
  // Persistent: one launch for every phase; otherwise one launch per phase (the counters
  // are then satisfied by stream order, and each list is balanced on its own).
  const int step = dt.tc_persistent ? nq : 1;
  for (int q0 = 0; q0 < nq; q0 += step) {
    const cudaError_t e =
        plan.ns_dtype == 2
            ? launch_impl<kShapePair, kVarSplit>(plan, dt, ws, ns_steps, q0, q0 + step, budget, ap, st)
        : dt.tc_shape == kShapePair
            ? launch_impl<kShapePair>(plan, dt, ws, ns_steps, q0, q0 + step, budget, ap, st)
        : dt.tc_shape == kShapePairWide
            ? launch_impl<kShapePairWide>(plan, dt, ws, ns_steps, q0, q0 + step, budget, ap, st)
            : launch_impl<kShapeSingle>(plan, dt, ws, ns_steps, q0, q0 + step, budget, ap, st);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_selftest_timeout(int* err, long long budget, cudaStream_t st) {
  selftest_timeout_kernel<<<1, 32, 0, st>>>(err, budget);
  return cudaGetLastError();
}

bool encode_tensor_maps(const Plan& plan, const void* ws, std::vector<CUtensorMap>* maps,
                        std::string* err) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (encode == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    const cudaError_t e =
        cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr) {
      *err = "cuTensorMapEncodeTiled is not available from the driver";
      return false;
    }
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  maps->assign(plan.mats.size() * kMapsPerMat, CUtensorMap{});
  const uint8_t* base = static_cast<const uint8_t*>(ws);
  const bool split = plan.ns_dtype == 2;  // three bf16 arrays per buffer, else one
  const uint64_t esz = 2;
  auto make = [&](CUtensorMap* m, int64_t off, uint64_t inner, uint64_t outer, uint64_t pitch,
                  uint32_t box_inner, uint32_t box_outer,
                  CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) -> bool {
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {pitch * esz};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    const CUresult r = encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                              const_cast<uint8_t*>(base + off), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
      char buf[160];
      std::snprintf(buf, sizeof(buf), "cuTensorMapEncodeTiled failed (%d) for a %llux%llu tensor",
                    (int)r, (unsigned long long)outer, (unsigned long long)inner);
      *err = buf;
      return false;
    }
    return true;
  };
  for (size_t i = 0; i < plan.mats.size(); ++i) {
    const MatDev& mt = plan.mats[i];
    CUtensorMap* m = maps->data() + i * kMapsPerMat;
    const int64_t xs[2] = {mt.x0, mt.x1};
    if (split) {
      // The same operand boxes as the bf16 path for each of the h, m and l arrays
      // (slot + part * kMapPart); the epilogue writes with plain stores.
      const int64_t xp = split_part_bytes((int64_t)mt.rows * mt.ldx * 2);
      const int64_t ap = split_part_bytes((int64_t)mt.m * mt.lda * 2);
      for (int part = 0; part < 3; ++part) {
        CUtensorMap* mp = m + part * kMapPart;
        for (int b = 0; b < 2; ++b) {
          const int64_t o = xs[b] + part * xp;
          if (!make(mp + 3 * b + 0, o, mt.cols, mt.rows, mt.ldx, 64, 128)) return false;
          if (!make(mp + 3 * b + 1, o, mt.cols, mt.rows, mt.ldx, 64, 256)) return false;
          if (!make(mp + 3 * b + 2, o, mt.cols, mt.rows, mt.ldx, 64, 64)) return false;
        }
        const int64_t ao = mt.a + part * ap, bo = mt.b + part * ap;
        if (!make(mp + kMapAK128, ao, mt.m, mt.m, mt.lda, 64, 128)) return false;
        if (!make(mp + kMapAK256, ao, mt.m, mt.m, mt.lda, 64, 256)) return false;
        if (!make(mp + kMapBK128, bo, mt.m, mt.m, mt.lda, 64, 128)) return false;
        if (!make(mp + kMapBK256, bo, mt.m, mt.m, mt.lda, 64, 256)) return false;
      }
      continue;
    }
    for (int b = 0; b < 2; ++b) {
      if (!make(m + 3 * b + 0, xs[b], mt.cols, mt.rows, mt.ldx, 64, 128)) return false;
      if (!make(m + 3 * b + 1, xs[b], mt.cols, mt.rows, mt.ldx, 64, 256)) return false;
      if (!make(m + 3 * b + 2, xs[b], mt.cols, mt.rows, mt.ldx, 64, 64)) return false;
    }
    if (!make(m + kMapAK128, mt.a, mt.m, mt.m, mt.lda, 64, 128)) return false;
    if (!make(m + kMapAK256, mt.a, mt.m, mt.m, mt.lda, 64, 256)) return false;
    if (!make(m + kMapBK128, mt.b, mt.m, mt.m, mt.lda, 64, 128)) return false;
    if (!make(m + kMapBK256, mt.b, mt.m, mt.m, mt.lda, 64, 256)) return false;
    const CUtensorMapSwizzle s64 = CU_TENSOR_MAP_SWIZZLE_64B;
    if (!make(m + kMapX0St, mt.x0, mt.cols, mt.rows, mt.ldx, 32, 32, s64)) return false;
    if (!make(m + kMapX1St, mt.x1, mt.cols, mt.rows, mt.ldx, 32, 32, s64)) return false;
    if (!make(m + kMapASt, mt.a, mt.m, mt.m, mt.lda, 32, 32, s64)) return false;
    if (!make(m + kMapBSt, mt.b, mt.m, mt.m, mt.lda, 32, 32, s64)) return false;
  }
  return true;
}

}  // namespace muon
