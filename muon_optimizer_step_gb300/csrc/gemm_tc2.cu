// bf16 Newton-Schulz phases on CTA pairs: tcgen05.mma.cta_group::2, 256 x 256 tiles.
//
// Same three phases and epilogues as the single-CTA kernel (Gram, Poly, Update of the
// quintic Newton-Schulz iteration, symmetric outputs computed on upper tiles and
// mirrored, 1/||X|| folded into the first iteration's epilogues), but every output tile
// of 256 x 256 is computed by a cluster of two CTAs on one TPC:
//   * CTA r of the pair loads rows [128r, 128r+128) of the tile's A operand and rows
//     [128r, 128r+128) of its B operand (half of N), 32 KB per 64-deep k-block;
//   * the even CTA issues tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 16), which
//     reads A and B from both CTAs' shared memory and accumulates into both CTAs' TMEM
//     (CTA r holds output rows [128r, 128r+128), all 256 columns);
//   * each CTA's four epilogue warps drain their own TMEM.
// Per SM this halves the B-operand traffic of a 128 x 256 single-CTA tile (32 KB instead
// of 48 KB per k-block for the same MMA work).
//
// Synchronisation: the even CTA's full[s] barrier takes one arrival (the even producer,
// announcing both CTAs' bytes) and both CTAs' copies; the MMA commit multicasts to both
// CTAs' empty[s] and acc_full[b]; acc_empty[b] of the even CTA counts one arrival per
// epilogue warp of the pair (8).  Every wait is bounded.
#include <cstdio>
#include <string>
#include <vector>

#include <cudaTypedefs.h>

#include "device_common.cuh"
#include "kernels.h"

namespace muon {

namespace {

constexpr int BM = 256, BN = 256, BK = kTcBK;   // pair tile
constexpr int HM = 128;                         // rows per CTA (of A and of B)
constexpr int STAGES = 7;
constexpr int UMMA_K = 16;
constexpr int A_BYTES = HM * BK * 2;            // 16 KB
constexpr int B_BYTES = HM * BK * 2;            // 16 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;  // 32 KB per CTA
constexpr int MN_BOX_BYTES = 64 * BK * 2;       // 8 KB
constexpr int NUM_THREADS = 384;  // warps 0-3 roles, warps 4-11 epilogue
constexpr int EPI_WARPS = 8;
constexpr int TMEM_COLS = 512;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256;
constexpr float kA = 3.4445f, kB = -4.7750f, kC = 2.0315f;

struct Tc2Params {
  const TileDev* tiles;
  const int32_t* cta_begin;  // per pair
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

struct TileOps {
  int a_map, b_map;
  int a_mn, b_mn;
};

__device__ __forceinline__ TileOps tile_ops(const MatDev& mt, int phase, int x_in) {
  const int xk = x_in ? kMapX1K128 : kMapX0K128;
  const int xmn = x_in ? kMapX1MN : kMapX0MN;
  TileOps o;
  if (phase == kPhaseGram) {
    if (mt.tall) { o.a_map = xmn; o.b_map = xmn; o.a_mn = 1; o.b_mn = 1; }
    else { o.a_map = xk; o.b_map = xk; o.a_mn = 0; o.b_mn = 0; }
  } else if (phase == kPhasePoly) {
    o.a_map = kMapAK128; o.b_map = kMapAK128; o.a_mn = 0; o.b_mn = 0;
  } else {
    if (mt.tall) { o.a_map = xk; o.b_map = kMapBK128; o.a_mn = 0; o.b_mn = 0; }
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

// Epilogue of accumulator columns [jb, jb+32) of output row i (same rules as the
// single-CTA kernel: Update writes a*X + acc scaled; symmetric phases write j >= i and
// the mirror (j, i)).
__device__ __forceinline__ void epilogue_chunk(const Tc2Params& p, const MatDev& mt, int i,
                                               int jb, const uint32_t (&acc)[32], float s) {
  float f[32];
  if (p.phase == kPhaseUpdate) {
    if (i >= mt.rows || jb >= mt.cols) return;
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

// Bounded wait that also tells the peer CTA to stop when it gives up.
__device__ __forceinline__ bool wait_pair(uint64_t* bar, uint32_t parity, const Tc2Params& p,
                                          volatile int* abort, uint32_t peer_abort) {
  if (mbar_wait_bounded(bar, parity, p.budget, p.err, abort)) return true;
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(peer_abort), "r"(1) : "memory");
  return false;
}

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

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
    ns_phase_tc2_kernel(const __grid_constant__ Tc2Params p) {
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
  const uint32_t rank = cluster_ctarank();  // 0: the CTA that issues the MMAs
  const int pair = blockIdx.x >> 1;
  const int t_begin = p.cta_begin[pair], t_end = p.cta_begin[pair + 1];
  const uint32_t peer_abort = mapa_shared(smem_u32(&abort_flag), rank ^ 1u);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);   // the even CTA's arrival, expecting both CTAs' bytes
      mbar_init(&empty[s], 1);  // the MMA commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 2 * EPI_WARPS);  // one arrival per epilogue warp of the pair
    }
    mbar_init(mma_done, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc_pair(tmem_slot, TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  volatile int* abort = &abort_flag;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer (both CTAs)
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
        const int ia = tile.i0 + HM * (int)rank;
        const int jb = tile.j0 + HM * (int)rank;
        bool ok = true;
        for (int kb = 0; kb < tile.kblocks; ++kb) {
          if (!wait_pair(&empty[stage], ph ^ 1u, p, abort, peer_abort)) {
            ok = false;
            break;
          }
          const uint32_t sa = smem_u32(tiles_smem + stage * STAGE_BYTES);
          const uint32_t sb = sa + A_BYTES;
          const uint32_t fbar = mapa_shared(smem_u32(&full[stage]), 0);
          const int k0 = kb * BK;
          // Only the even CTA arrives, announcing both CTAs' bytes; the odd CTA's copies may
          // land first (the transaction count then dips below zero, which mbarriers allow,
          // and the phase still needs the even CTA's arrival to complete).
          if (rank == 0) mbar_arrive_expect_tx(&full[stage], 2 * STAGE_BYTES);
          if (ops.a_mn) {
            tma_load_2d_pair(sa, amap, ia, k0, fbar);
            tma_load_2d_pair(sa + MN_BOX_BYTES, amap, ia + 64, k0, fbar);
          } else {
            tma_load_2d_pair(sa, amap, k0, ia, fbar);
          }
          if (ops.b_mn) {
            tma_load_2d_pair(sb, bmap, jb, k0, fbar);
            tma_load_2d_pair(sb + MN_BOX_BYTES, bmap, jb + 64, k0, fbar);
          } else {
            tma_load_2d_pair(sb, bmap, k0, jb, fbar);
          }
          ++nfill;
          if (++stage == STAGES) {
            stage = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
      }
      // The even CTA's full barriers count both CTAs' copies: drain them there.
      if (rank == 0)
        for (long long k = nfill - 1; k >= 0 && k >= nfill - STAGES; --k)
          wait_drain(&full[k % STAGES], (uint32_t)((k / STAGES) & 1), p.budget, p.err);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer (even CTA)
    if (lane == 0 && rank == 0) {
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
        if (!wait_pair(&acc_empty[ab], (uint32_t)(((lt >> 1) & 1) ^ 1), p, abort, peer_abort))
          break;
        tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(ab * BN);
        bool ok = true;
        for (int kb = 0; kb < tile.kblocks; ++kb) {
          if (!wait_pair(&full[stage], ph, p, abort, peer_abort)) {
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
            tc_mma_f16_pair(d, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          tc_commit_pair(&empty[stage], (uint16_t)0x3);
          if (++stage == STAGES) {
            stage = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit_pair(&acc_full[ab], (uint16_t)0x3);
      }
      tc_commit_pair(mma_done, (uint16_t)0x1);
      wait_drain(mma_done, 0, p.budget, p.err);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- epilogue (both CTAs)
    // Two epilogue warps per TMEM lane quarter (warp % 4), each draining half the columns.
    const int q = warp & 3;
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
      if (!__all_sync(0xffffffffu, ok)) {
        asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(peer_abort), "r"(1) : "memory");
        break;
      }
      tc_fence_after();
      float s = 1.f;
      if (p.iter0 && p.phase != kPhasePoly) {
        const float inv = p.inv_norm[tile.mat];
        s = p.phase == kPhaseGram ? inv * inv : inv;
      }
      const int i = tile.i0 + HM * (int)rank + r;
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
      if (lane == 0) {
        if (rank == 0) mbar_arrive(&acc_empty[ab]);
        else mbar_arrive_cluster(mapa_shared(smem_u32(&acc_empty[ab]), 0));
      }
    }
  }
  tc_fence_before();
  cluster_sync();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

}  // namespace

cudaError_t prepare_tc2_kernel(int* max_pairs) {
  cudaError_t e = cudaFuncSetAttribute(ns_phase_tc2_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * 1024, 1, 1);
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  int n = 0;
  e = cudaOccupancyMaxActiveClusters(&n, ns_phase_tc2_kernel, &cfg);
  if (e != cudaSuccess) return e;
  *max_pairs = n;
  return cudaSuccess;
}

cudaError_t launch_ns_phase_tc2(const Plan& plan, const DevTables& dt, void* ws, int phase,
                                int x_in, int iter0, long long budget, const ApplyArgs* ap,
                                cudaStream_t st) {
  const int pairs = dt.grid[phase];
  if (pairs == 0) return cudaSuccess;
  uint8_t* w = static_cast<uint8_t*>(ws);
  Tc2Params p;
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
  ns_phase_tc2_kernel<<<2 * pairs, NUM_THREADS, SMEM_BYTES, st>>>(p);
  return cudaGetLastError();
}

}  // namespace muon
