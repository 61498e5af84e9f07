// fp32 Newton-Schulz phases on the CUDA cores (the precision path of the Muon step).
//
// One launch runs one phase of one Newton-Schulz iteration for every matrix of the flat
// buffer (a grouped, persistent launch over a host-planned tile list):
//   Gram    A = X X^T          (tall: A = X^T X), upper-triangle tiles, mirrored;
//   Poly    B = b*A + c*A A    (A symmetric), upper-triangle tiles, mirrored;
//   Update  X' = s*(a*X + B X) (tall: X' = s*(a*X + X B)),
// with s = 1/||X||_F on the first iteration (the normalisation folded into the epilogue;
// the Gram epilogue takes s^2) and (a, b, c) = (3.4445, -4.7750, 2.0315).
// 128 x 128 output tiles, 16-deep k-slices staged in shared memory, 8 x 8 per thread.
#include "device_common.cuh"
#include "kernels.h"

namespace muon {

namespace {

constexpr int BM = kF32BM, BN = kF32BN, BK = 16, PAD = 4, NT = 256;
constexpr float kA = 3.4445f, kB = -4.7750f, kC = 2.0315f;

struct OpDesc {
  const float* base;
  int ld;
  int mn;       // extent along the operand's M (or N) index
  int mn_major; // 0: element (i, k) at base[i*ld + k]; 1: at base[k*ld + i]
};

// Loads the BK x 128 slice [k0, k0+BK) x [i0, i0+128) of an operand into registers.
__device__ __forceinline__ void load_slice(const OpDesc& op, int i0, int k0, int K,
                                           float (&r)[8]) {
  const int t = threadIdx.x;
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int idx = t + NT * q;
    if (!op.mn_major) {
      const int row = idx >> 2, kq = idx & 3;
      const int gi = i0 + row, gk = k0 + 4 * kq;
      if (gi < op.mn && gk + 3 < K) {
        const float4 v = *reinterpret_cast<const float4*>(op.base + (int64_t)gi * op.ld + gk);
        r[4 * q + 0] = v.x; r[4 * q + 1] = v.y; r[4 * q + 2] = v.z; r[4 * q + 3] = v.w;
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          r[4 * q + e] = (gi < op.mn && gk + e < K) ? op.base[(int64_t)gi * op.ld + gk + e] : 0.f;
      }
    } else {
      const int kk = idx >> 5, iq = idx & 31;
      const int gk = k0 + kk, gi = i0 + 4 * iq;
      if (gk < K && gi + 3 < op.mn) {
        const float4 v = *reinterpret_cast<const float4*>(op.base + (int64_t)gk * op.ld + gi);
        r[4 * q + 0] = v.x; r[4 * q + 1] = v.y; r[4 * q + 2] = v.z; r[4 * q + 3] = v.w;
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          r[4 * q + e] = (gk < K && gi + e < op.mn) ? op.base[(int64_t)gk * op.ld + gi + e] : 0.f;
      }
    }
  }
}

__device__ __forceinline__ void store_slice(const OpDesc& op, const float (&r)[8],
                                            float (*s)[BM + PAD]) {
  const int t = threadIdx.x;
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int idx = t + NT * q;
    if (!op.mn_major) {
      const int row = idx >> 2, kq = idx & 3;
#pragma unroll
      for (int e = 0; e < 4; ++e) s[4 * kq + e][row] = r[4 * q + e];
    } else {
      const int kk = idx >> 5, iq = idx & 31;
      *reinterpret_cast<float4*>(&s[kk][4 * iq]) =
          make_float4(r[4 * q + 0], r[4 * q + 1], r[4 * q + 2], r[4 * q + 3]);
    }
  }
}

__global__ void __launch_bounds__(NT)
ns_phase_f32_kernel(const TileDev* __restrict__ tiles, const int32_t* __restrict__ cta_begin,
                    const MatDev* __restrict__ mats, uint8_t* __restrict__ ws,
                    const float* __restrict__ inv_norm, int phase, int x_in, int iter0,
                    int64_t n_tiles, const DebugCtx dbg) {
  __shared__ __align__(16) float As[BK][BM + PAD];
  __shared__ __align__(16) float Bs[BK][BN + PAD];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  if (debug_halted(dbg)) return;
  if (kDebugChecks) {
    const int b0 = cta_begin[blockIdx.x], b1 = cta_begin[blockIdx.x + 1];
    if (b0 < 0 || b1 < b0 || b1 > n_tiles) {
      if (threadIdx.x == 0) debug_fail(dbg);
      return;
    }
  }
  for (int ti = cta_begin[blockIdx.x]; ti < cta_begin[blockIdx.x + 1]; ++ti) {
    const TileDev tile = tiles[ti];
    if (kDebugChecks && !debug_tile_ok(tile, phase, mats, dbg, BM, BN, BK)) {
      if (threadIdx.x == 0) debug_fail(dbg);
      continue;
    }
    const MatDev mt = mats[tile.mat];
    const float* xin = reinterpret_cast<const float*>(ws + (x_in ? mt.x1 : mt.x0));
    float* xout = reinterpret_cast<float*>(ws + (x_in ? mt.x0 : mt.x1));
    float* am = reinterpret_cast<float*>(ws + mt.a);
    float* bm = reinterpret_cast<float*>(ws + mt.b);
    OpDesc opa, opb;
    int K;
    if (phase == kPhaseGram) {
      opa = {xin, mt.ldx, mt.m, mt.tall};
      opb = opa;
      K = mt.n;
    } else if (phase == kPhasePoly) {
      opa = {am, mt.lda, mt.m, 0};
      opb = opa;
      K = mt.m;
    } else if (!mt.tall) {
      opa = {bm, mt.lda, mt.m, 0};
      opb = {xin, mt.ldx, mt.cols, 1};
      K = mt.m;
    } else {
      opa = {xin, mt.ldx, mt.rows, 0};
      opb = {bm, mt.lda, mt.m, 0};
      K = mt.m;
    }
    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
    float ra[8], rb[8];
    load_slice(opa, tile.i0, 0, K, ra);
    load_slice(opb, tile.j0, 0, K, rb);
    for (int k0 = 0; k0 < K; k0 += BK) {
      __syncthreads();
      store_slice(opa, ra, As);
      store_slice(opb, rb, Bs);
      __syncthreads();
      if (k0 + BK < K) {
        load_slice(opa, tile.i0, k0 + BK, K, ra);
        load_slice(opb, tile.j0, k0 + BK, K, rb);
      }
#pragma unroll
      for (int kk = 0; kk < BK; ++kk) {
        const float4 a0 = *reinterpret_cast<const float4*>(&As[kk][ty * 4]);
        const float4 a1 = *reinterpret_cast<const float4*>(&As[kk][64 + ty * 4]);
        const float4 b0 = *reinterpret_cast<const float4*>(&Bs[kk][tx * 4]);
        const float4 b1 = *reinterpret_cast<const float4*>(&Bs[kk][64 + tx * 4]);
        const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
        const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
      }
    }
    // Epilogue.
    const float s = iter0 ? inv_norm[tile.mat] : 1.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int gi = tile.i0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + (i - 4));
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int gj = tile.j0 + (j < 4 ? tx * 4 + j : 64 + tx * 4 + (j - 4));
        if (phase == kPhaseUpdate) {
          if (gi < mt.rows && gj < mt.cols) {
            const int64_t o = (int64_t)gi * mt.ldx + gj;
            xout[o] = s * fmaf(kA, xin[o], acc[i][j]);
          }
        } else if (gi < mt.m && gj < mt.m && gj >= gi) {
          float v;
          float* out;
          if (phase == kPhaseGram) {
            v = acc[i][j] * (s * s);
            out = am;
          } else {
            v = fmaf(kB, am[(int64_t)gi * mt.lda + gj], kC * acc[i][j]);
            out = bm;
          }
          out[(int64_t)gi * mt.lda + gj] = v;
          if (gj != gi) out[(int64_t)gj * mt.lda + gi] = v;
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_ns_phase_f32(const Plan& plan, const DevTables& dt, void* ws, int phase,
                                int x_in, int iter0, cudaStream_t st) {
  const int grid = dt.grid[phase];
  if (grid == 0) return cudaSuccess;
  uint8_t* w = static_cast<uint8_t*>(ws);
  ns_phase_f32_kernel<<<grid, NT, 0, st>>>(dt.tiles[phase], dt.cta_begin[phase], dt.mats, w,
                                           reinterpret_cast<const float*>(w + plan.ws_inv_norm),
                                           phase, x_in, iter0, dt.n_tiles[phase],
                                           make_debug_ctx(plan, dt));
  return cudaGetLastError();
}

}  // namespace muon
