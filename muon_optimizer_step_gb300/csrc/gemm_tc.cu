// bf16 Newton-Schulz phases on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// One launch runs one phase of one Newton-Schulz iteration for every matrix of a flat
// buffer: a persistent, grouped launch whose CTAs walk host-planned tile lists.
//   Gram    A = X X^T           (tall X: A = X^T X)      upper-triangle tiles, mirrored
//   Poly    B = b*A + c*A A     (A symmetric)            upper-triangle tiles, mirrored
//   Update  X' = s*(a*X + B X)  (tall X: X' = s*(a*X + X B))
// s = 1/||X||_F on the first iteration and 1 after it (the Gram epilogue takes s^2), so the
// Frobenius normalisation costs no separate pass; (a, b, c) = (3.4445, -4.7750, 2.0315).
// X stays in its stored row-major orientation: the transposes a tall matrix needs are
// MN-major operand reads (the tcgen05 transpose bits), never data movement.
//
// CTA layout (256 threads, one CTA per SM):
//   warp 0      TMA producer: 128x64 A-slice + 256x64 B-slice per stage, SWIZZLE_128B
//   warp 1      MMA issuer: tcgen05.mma.cta_group::1.kind::f16, M=128 N=256 K=16
//   warp 2      TMEM allocator (512 columns = two 128x256 fp32 accumulators)
//   warps 4-7   epilogue: tcgen05.ld 32x32b, fused scaling / polynomial / update, stores
// Stages are handed over with mbarriers; every wait is bounded (see mbar_wait_bounded).
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include <cudaTypedefs.h>

#include "device_common.cuh"
#include "kernels.h"

namespace muon {

namespace {

constexpr int BM = kTcBM, BN = kTcBN, BK = kTcBK;
constexpr int STAGES = 4;
constexpr int UMMA_K = 16;
constexpr int A_BYTES = BM * BK * 2;                  // 16 KB
constexpr int B_BYTES = BN * BK * 2;                  // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;        // 48 KB
constexpr int MN_BOX_BYTES = 64 * BK * 2;             // one 64 (mn) x 64 (k) box: 8 KB
constexpr int NUM_THREADS = 384;  // warps 0-3 roles, warps 4-11 epilogue
constexpr int EPI_WARPS = 8;
constexpr int TMEM_COLS = 512;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 /*align*/ + 256 /*barriers*/;
constexpr float kA = 3.4445f, kB = -4.7750f, kC = 2.0315f;

struct TcParams {
  const TileDev* tiles;
  const int32_t* cta_begin;
  const MatDev* mats;
  const CUtensorMap* tmaps;
  uint8_t* ws;
  const float* inv_norm;
  int* err;
  long long budget;
  int phase;
  int x_in;
  int iter0;
  int apply;        // last Update: also W <- W*decay - lr*scale*O (fp32 O)
  ApplyArgs ap;
};

// Which tensor maps, transpose bits and reduction length a tile of `phase` uses.
struct TileOps {
  int a_map, b_map;  // map slots
  int a_mn, b_mn;    // 1: MN-major operand (loaded as 64-wide boxes)
  int K;
};

__device__ __forceinline__ TileOps tile_ops(const MatDev& mt, int phase, int x_in) {
  const int xk128 = x_in ? kMapX1K128 : kMapX0K128;
  const int xk256 = x_in ? kMapX1K256 : kMapX0K256;
  const int xmn = x_in ? kMapX1MN : kMapX0MN;
  TileOps o;
  if (phase == kPhaseGram) {
    o.K = mt.n;
    if (mt.tall) { o.a_map = xmn; o.b_map = xmn; o.a_mn = 1; o.b_mn = 1; }
    else { o.a_map = xk128; o.b_map = xk256; o.a_mn = 0; o.b_mn = 0; }
  } else if (phase == kPhasePoly) {
    o.K = mt.m;
    o.a_map = kMapAK128; o.b_map = kMapAK256; o.a_mn = 0; o.b_mn = 0;
  } else {
    o.K = mt.m;
    if (mt.tall) { o.a_map = xk128; o.b_map = kMapBK256; o.a_mn = 0; o.b_mn = 0; }
    else { o.a_map = kMapBK128; o.b_map = xmn; o.a_mn = 0; o.b_mn = 1; }
  }
  return o;
}

__device__ __forceinline__ void store_bf16x32(__nv_bfloat16* dst, const float (&f)[32]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 u;
    u.x = pack_bf16x2(f[8 * q + 0], f[8 * q + 1]);
    u.y = pack_bf16x2(f[8 * q + 2], f[8 * q + 3]);
    u.z = pack_bf16x2(f[8 * q + 4], f[8 * q + 5]);
    u.w = pack_bf16x2(f[8 * q + 6], f[8 * q + 7]);
    reinterpret_cast<uint4*>(dst)[q] = u;
  }
}

__device__ __forceinline__ void load_bf16x32(const __nv_bfloat16* src, float (&f)[32]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 u = reinterpret_cast<const uint4*>(src)[q];
    f[8 * q + 0] = bf16_lo(u.x); f[8 * q + 1] = bf16_hi(u.x);
    f[8 * q + 2] = bf16_lo(u.y); f[8 * q + 3] = bf16_hi(u.y);
    f[8 * q + 4] = bf16_lo(u.z); f[8 * q + 5] = bf16_hi(u.z);
    f[8 * q + 6] = bf16_lo(u.w); f[8 * q + 7] = bf16_hi(u.w);
  }
}

// Epilogue of 32 consecutive accumulator columns [jb, jb+32) of output row i.
__device__ __forceinline__ void epilogue_chunk(const TcParams& p, const MatDev& mt, int i,
                                               int jb, const uint32_t (&acc)[32], float s) {
  float f[32];
  if (p.phase == kPhaseUpdate) {
    if (i >= mt.rows) return;
    const __nv_bfloat16* xin =
        reinterpret_cast<const __nv_bfloat16*>(p.ws + (p.x_in ? mt.x1 : mt.x0));
    __nv_bfloat16* xout = reinterpret_cast<__nv_bfloat16*>(p.ws + (p.x_in ? mt.x0 : mt.x1));
    const int64_t row = (int64_t)i * mt.ldx;
    if (jb + 32 <= mt.cols) {
      float x[32];
      load_bf16x32(xin + row + jb, x);
      if (p.apply) {
        // Issue the weight loads with the X loads, before any store, so that the two
        // memory round trips of this chunk overlap.
        float w[32];
        const bool vec = apply_load_row_run(p.ap, mt, i, jb, w);
#pragma unroll
        for (int t = 0; t < 32; ++t) f[t] = s * fmaf(kA, x[t], __uint_as_float(acc[t]));
        store_bf16x32(xout + row + jb, f);
        apply_store_row_run(p.ap, mt, i, jb, vec, w, f);
        return;
      }
#pragma unroll
      for (int t = 0; t < 32; ++t) f[t] = s * fmaf(kA, x[t], __uint_as_float(acc[t]));
      store_bf16x32(xout + row + jb, f);
    } else {
#pragma unroll
      for (int t = 0; t < 32; ++t) {
        const int j = jb + t;
        f[t] = 0.f;
        if (j < mt.cols) {
          f[t] = s * fmaf(kA, __bfloat162float(xin[row + j]), __uint_as_float(acc[t]));
          xout[row + j] = __float2bfloat16_rn(f[t]);
        }
      }
    }
    if (p.apply) apply_row_run(p.ap, mt, i, jb, min(32, mt.cols - jb), f);
    return;
  }
  // Symmetric outputs (A or B, m x m): write (i, j) for j >= i and its mirror (j, i).
  if (i >= mt.m || jb + 31 < i || jb >= mt.m) return;
  __nv_bfloat16* am = reinterpret_cast<__nv_bfloat16*>(p.ws + mt.a);
  __nv_bfloat16* out = p.phase == kPhaseGram ? am : reinterpret_cast<__nv_bfloat16*>(p.ws + mt.b);
  const int64_t row = (int64_t)i * mt.lda;
  const bool full = (jb + 32 <= mt.m);
  if (p.phase == kPhaseGram) {
#pragma unroll
    for (int t = 0; t < 32; ++t) f[t] = __uint_as_float(acc[t]) * s;
  } else if (full) {
    float a[32];
    load_bf16x32(am + row + jb, a);
#pragma unroll
    for (int t = 0; t < 32; ++t) f[t] = fmaf(kB, a[t], kC * __uint_as_float(acc[t]));
  } else {
#pragma unroll
    for (int t = 0; t < 32; ++t) {
      const int j = jb + t;
      f[t] = j < mt.m ? fmaf(kB, __bfloat162float(am[row + j]), kC * __uint_as_float(acc[t]))
                      : 0.f;
    }
  }
  if (full && jb >= i) {
    store_bf16x32(out + row + jb, f);
  } else {
#pragma unroll
    for (int t = 0; t < 32; ++t) {
      const int j = jb + t;
      if (j >= i && j < mt.m) out[row + j] = __float2bfloat16_rn(f[t]);
    }
  }
#pragma unroll
  for (int t = 0; t < 32; ++t) {
    const int j = jb + t;
    if (j > i && j < mt.m) out[(int64_t)j * mt.lda + i] = __float2bfloat16_rn(f[t]);
  }
}

// Like mbar_wait_bounded but ignores the abort flag: used to drain copies and MMAs that
// are already in flight before the block exits.
__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity, long long budget,
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

__global__ void __launch_bounds__(NUM_THREADS, 1) ns_phase_tc_kernel(const __grid_constant__ TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ int abort_flag;
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* tiles_smem = smem_raw + pad;
  uint64_t* bars = reinterpret_cast<uint64_t*>(tiles_smem + STAGES * STAGE_BYTES);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* acc_full = bars + 2 * STAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* mma_done = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t_begin = p.cta_begin[blockIdx.x], t_end = p.cta_begin[blockIdx.x + 1];

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], EPI_WARPS);  // one arrival per epilogue warp
    }
    mbar_init(mma_done, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  volatile int* abort = &abort_flag;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t ph = 0;
      long long nfill = 0;
      for (int ti = t_begin; ti < t_end; ++ti) {
        const TileDev tile = p.tiles[ti];
        const MatDev& mt = p.mats[tile.mat];
        const TileOps ops = tile_ops(mt, p.phase, p.x_in);
        const CUtensorMap* amap = p.tmaps + (size_t)tile.mat * kMapsPerMat + ops.a_map;
        const CUtensorMap* bmap = p.tmaps + (size_t)tile.mat * kMapsPerMat + ops.b_map;
        bool ok = true;
        for (int kb = 0; kb < tile.kblocks; ++kb) {
          if (!mbar_wait_bounded(&empty[stage], ph ^ 1u, p.budget, p.err, abort)) {
            ok = false;
            break;
          }
          uint8_t* sa = tiles_smem + stage * STAGE_BYTES;
          uint8_t* sb = sa + A_BYTES;
          mbar_arrive_expect_tx(&full[stage], STAGE_BYTES);
          const int k0 = kb * BK;
          if (ops.a_mn) {
            tma_load_2d(sa, amap, tile.i0, k0, &full[stage]);
            tma_load_2d(sa + MN_BOX_BYTES, amap, tile.i0 + 64, k0, &full[stage]);
          } else {
            tma_load_2d(sa, amap, k0, tile.i0, &full[stage]);
          }
          if (ops.b_mn) {
#pragma unroll
            for (int q = 0; q < 4; ++q)
              tma_load_2d(sb + q * MN_BOX_BYTES, bmap, tile.j0 + 64 * q, k0, &full[stage]);
          } else {
            tma_load_2d(sb, bmap, k0, tile.j0, &full[stage]);
          }
          ++nfill;
          if (++stage == STAGES) {
            stage = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
      }
      // Every copy issued must land before the block exits (already true unless aborted).
      for (long long k = nfill - 1; k >= 0 && k >= nfill - STAGES; --k)
        mbar_wait_drain(&full[k % STAGES], (uint32_t)((k / STAGES) & 1), p.budget, p.err);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t ph = 0;
      int lt = 0;
      const uint32_t sbase = smem_u32(tiles_smem);
      for (int ti = t_begin; ti < t_end; ++ti, ++lt) {
        const TileDev tile = p.tiles[ti];
        const MatDev& mt = p.mats[tile.mat];
        const TileOps ops = tile_ops(mt, p.phase, p.x_in);
        const uint32_t idesc = idesc_bf16(BM, BN, ops.a_mn, ops.b_mn);
        const int ab = lt & 1;
        if (!mbar_wait_bounded(&acc_empty[ab], (uint32_t)(((lt >> 1) & 1) ^ 1), p.budget, p.err,
                               abort))
          break;
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(ab * BN);
        bool ok = true;
        for (int kb = 0; kb < tile.kblocks; ++kb) {
          if (!mbar_wait_bounded(&full[stage], ph, p.budget, p.err, abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = sbase + stage * STAGE_BYTES;
          const uint32_t sb = sa + A_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / UMMA_K; ++kk) {
            const uint64_t ad = ops.a_mn ? smem_desc_sw128(sa + kk * 2048, MN_BOX_BYTES, 1024)
                                         : smem_desc_sw128(sa + kk * 32, 16, 1024);
            const uint64_t bd = ops.b_mn ? smem_desc_sw128(sb + kk * 2048, MN_BOX_BYTES, 1024)
                                         : smem_desc_sw128(sb + kk * 32, 16, 1024);
            tc_mma_f16(d, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          tc_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(&acc_full[ab]);
      }
      // Every MMA issued must complete before TMEM is released.
      tc_commit(mma_done);
      mbar_wait_drain(mma_done, 0, p.budget, p.err);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- epilogue
    // Two epilogue warps per TMEM lane quarter (warp % 4), each draining half the columns.
    const int q = warp & 3;  // TMEM lanes 32q .. 32q+31
    const int half = (warp - 4) >> 2;
    const int r = 32 * q + lane;
    int lt = 0;
    for (int ti = t_begin; ti < t_end; ++ti, ++lt) {
      if (__any_sync(0xffffffffu, *abort != 0)) break;
      const TileDev tile = p.tiles[ti];
      const MatDev& mt = p.mats[tile.mat];
      const int ab = lt & 1;
      const bool ok = mbar_wait_bounded(&acc_full[ab], (uint32_t)((lt >> 1) & 1), p.budget,
                                        p.err, abort);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      float s = 1.f;
      if (p.iter0 && p.phase != kPhasePoly) {
        const float inv = p.inv_norm[tile.mat];
        s = p.phase == kPhaseGram ? inv * inv : inv;
      }
      const int i = tile.i0 + r;
#pragma unroll 1
      for (int c = half * (BN / 64); c < (half + 1) * (BN / 64); ++c) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(ab * BN + 32 * c),
                           v);
        tmem_ld_wait();
        epilogue_chunk(p, mt, i, tile.j0 + 32 * c, v, s);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[ab]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
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

}  // namespace

cudaError_t prepare_tc_kernel() {
  return cudaFuncSetAttribute(ns_phase_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              SMEM_BYTES);
}

cudaError_t launch_ns_phase_tc(const Plan& plan, const DevTables& dt, void* ws, int phase,
                               int x_in, int iter0, long long budget, const ApplyArgs* ap,
                               cudaStream_t st) {
  const int grid = dt.grid[phase];
  if (grid == 0) return cudaSuccess;
  uint8_t* w = static_cast<uint8_t*>(ws);
  TcParams p;
  p.tiles = dt.tiles[phase];
  p.cta_begin = dt.cta_begin[phase];
  p.mats = dt.mats;
  p.tmaps = dt.tmaps;
  p.ws = w;
  p.inv_norm = reinterpret_cast<const float*>(w + plan.ws_inv_norm);
  p.err = dt.err;
  p.budget = budget;
  p.phase = phase;
  p.x_in = x_in;
  p.iter0 = iter0;
  p.apply = ap != nullptr ? 1 : 0;
  if (ap != nullptr) p.ap = *ap;
  ns_phase_tc_kernel<<<grid, NUM_THREADS, SMEM_BYTES, st>>>(p);
  return cudaGetLastError();
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
  auto make = [&](CUtensorMap* m, int64_t off, uint64_t inner, uint64_t outer, uint64_t pitch,
                  uint32_t box_inner, uint32_t box_outer) -> bool {
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {pitch * 2};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    const CUresult r = encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                              const_cast<uint8_t*>(base + off), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
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
    for (int b = 0; b < 2; ++b) {
      if (!make(m + 3 * b + 0, xs[b], mt.cols, mt.rows, mt.ldx, 64, BM)) return false;
      if (!make(m + 3 * b + 1, xs[b], mt.cols, mt.rows, mt.ldx, 64, BN)) return false;
      if (!make(m + 3 * b + 2, xs[b], mt.cols, mt.rows, mt.ldx, 64, 64)) return false;
    }
    if (!make(m + kMapAK128, mt.a, mt.m, mt.m, mt.lda, 64, BM)) return false;
    if (!make(m + kMapAK256, mt.a, mt.m, mt.m, mt.lda, 64, BN)) return false;
    if (!make(m + kMapBK128, mt.b, mt.m, mt.m, mt.lda, 64, BM)) return false;
    if (!make(m + kMapBK256, mt.b, mt.m, mt.m, mt.lda, 64, BN)) return false;
  }
  return true;
}

}  // namespace muon
