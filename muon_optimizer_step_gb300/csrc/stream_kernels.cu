// Streaming kernels of the Muon step: flat fp32 passes bound by HBM bandwidth.
//
//  * momentum_input: "Opt step" steps 1-3 of "Add initial Muon+M-FSDPv2 implementation"
//    (FsdpMuon._compute_momentum_inputs in the Megatron-Core API docs): M <- mu*M + G,
//    X = G + mu*M (Nesterov) or M, written at its row-major place in the matrix's full
//    buffer (the owner gather, as indexing), plus a per-chunk sum of X^2 for ||X||_F.
//  * apply: steps 5-6 (FsdpMuon._apply_local_updates): W <- W*(1 - lr*wd)
//    - lr*sqrt(max(1, rows/cols))*O, O read from the full buffer at each flat element's
//    place (the owner scatter, as indexing), W written in shard order.
//  * gather / scatter / export / full_input: the same index map as bit copies.
//
// Every kernel walks the chunk table: a chunk lies inside one matrix, at a fixed place of
// its row-major index.  Inside one shard a block reads it with 128-bit accesses; across a
// shard edge it reads it element by element, in the same per-thread order, so that the
// per-chunk sums of squares do not depend on how the buffer is sharded.
#include "device_common.cuh"
#include "kernels.h"

namespace muon {

namespace {

constexpr int kThreads = 256;
constexpr int kBlocksPerSm = 8;

__device__ __forceinline__ void store4(__nv_bfloat16* p, float a, float b, float c, float d) {
  uint2 u;
  u.x = pack_bf16x2(a, b);
  u.y = pack_bf16x2(c, d);
  *reinterpret_cast<uint2*>(p) = u;
}
__device__ __forceinline__ void store4(float* p, float a, float b, float c, float d) {
  *reinterpret_cast<float4*>(p) = make_float4(a, b, c, d);
}
__device__ __forceinline__ void store1(__nv_bfloat16* p, float a) { *p = __float2bfloat16_rn(a); }
__device__ __forceinline__ void store1(float* p, float a) { *p = a; }

__device__ __forceinline__ float4 load4(const __nv_bfloat16* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  return make_float4(bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y), bf16_hi(u.y));
}
__device__ __forceinline__ float4 load4(const float* p) {
  return *reinterpret_cast<const float4*>(p);
}
__device__ __forceinline__ float load1(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ float load1(const float* p) { return *p; }

// An X buffer of split fp32 values: the h array and the distance (elements) from each
// part's array to the next one's (h, m, l).
struct SplitPtr {
  __nv_bfloat16* h;
  int64_t part;
};
__device__ __forceinline__ SplitPtr operator+(SplitPtr a, int64_t k) { return {a.h + k, a.part}; }
__device__ __forceinline__ void store4(SplitPtr p, float a, float b, float c, float d) {
  const float v[4] = {a, b, c, d};
  __nv_bfloat16 q[3][4];
#pragma unroll
  for (int e = 0; e < 4; ++e) split_bf16x3(v[e], q[0][e], q[1][e], q[2][e]);
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    uint2 u;
    u.x = (uint32_t)__bfloat16_as_ushort(q[k][0]) | ((uint32_t)__bfloat16_as_ushort(q[k][1]) << 16);
    u.y = (uint32_t)__bfloat16_as_ushort(q[k][2]) | ((uint32_t)__bfloat16_as_ushort(q[k][3]) << 16);
    *reinterpret_cast<uint2*>(p.h + k * p.part) = u;
  }
}
__device__ __forceinline__ void store1(SplitPtr p, float a) {
  __nv_bfloat16 h, m, l;
  split_bf16x3(a, h, m, l);
  p.h[0] = h;
  p.h[p.part] = m;
  p.h[2 * p.part] = l;
}
__device__ __forceinline__ float4 load4(SplitPtr p) {
  const float4 h = load4(static_cast<const __nv_bfloat16*>(p.h));
  const float4 m = load4(static_cast<const __nv_bfloat16*>(p.h + p.part));
  const float4 l = load4(static_cast<const __nv_bfloat16*>(p.h + 2 * p.part));
  return make_float4(h.x + (m.x + l.x), h.y + (m.y + l.y), h.z + (m.z + l.z),
                     h.w + (m.w + l.w));
}
__device__ __forceinline__ float load1(SplitPtr p) {
  return __bfloat162float(p.h[0]) +
         (__bfloat162float(p.h[p.part]) + __bfloat162float(p.h[2 * p.part]));
}

// The X buffer at workspace byte offset `off` of matrix mt, as element type XT.
template <typename XT>
struct XBuf {
  using ptr = XT*;
  __device__ static ptr at(const uint8_t* ws, int64_t off, const MatDev&) {
    return reinterpret_cast<XT*>(const_cast<uint8_t*>(ws) + off);
  }
};
template <>
struct XBuf<Bf16x3> {
  using ptr = SplitPtr;
  __device__ static ptr at(const uint8_t* ws, int64_t off, const MatDev& mt) {
    return {reinterpret_cast<__nv_bfloat16*>(const_cast<uint8_t*>(ws) + off),
            split_part_bytes((int64_t)mt.rows * mt.ldx * 2) / 2};
  }
};

// Fixed-shape block sum (same order every run); the result is valid in thread 0.
__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  float s = 0.f;
  if (w == 0) {
    s = (l < kThreads / 32) ? red[l] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  }
  return s;
}

// Sum-of-squares updates with explicit rounding (no FMA contraction), so that the
// 128-bit path and the per-element path add the same terms in the same order.
__device__ __forceinline__ float add_sq4(float ss, float a, float b, float c, float d) {
  return __fadd_rn(ss, __fadd_rn(__fadd_rn(__fmul_rn(a, a), __fmul_rn(b, b)),
                                 __fadd_rn(__fmul_rn(c, c), __fmul_rn(d, d))));
}
__device__ __forceinline__ float add_sq1(float ss, float a) { return __fadd_rn(ss, __fmul_rn(a, a)); }

// Element t of a chunk in the shards (a chunk may cross shard edges).
__device__ __forceinline__ float* elem_ptr(const ShardPtrs& P, const ChunkDev& ch, int64_t L,
                                           int64_t t) {
  int64_t o = ch.shard_off + t;
  int s = ch.shard;
  if (o >= L) {
    const int64_t q = o / L;
    s += (int)q;
    o -= q * L;
  }
  return P.p[s] + o;
}

// Position of row-major element `local` of a matrix in its pitched X buffer.
__device__ __forceinline__ int64_t x_index(const MatDev& mt, int64_t local) {
  if (mt.ldx == mt.cols) return local;
  const int64_t r = local / mt.cols;
  return r * mt.ldx + (local - r * mt.cols);
}

template <typename XT>
__global__ void __launch_bounds__(kThreads)
momentum_input_kernel(const ChunkDev* __restrict__ chunks, int64_t n_chunks,
                      const MatDev* __restrict__ mats, ShardPtrs G, ShardPtrs M, int64_t L,
                      uint8_t* __restrict__ ws, float* __restrict__ partials,
                      const __grid_constant__ GroupParams gp, const DebugCtx dbg) {
  __shared__ float red[32];
  if (debug_halted(dbg)) return;
  for (int64_t ci = blockIdx.x; ci < n_chunks; ci += gridDim.x) {
    const ChunkDev ch = chunks[ci];
    if (kDebugChecks && (!debug_chunk_ok(ch, mats, dbg, &G) || !debug_chunk_ok(ch, mats, dbg, &M)))
      continue;
    const MatDev& mt = mats[ch.mat];
    const float mu = gp.mu[mt.group];
    const int nesterov = gp.nesterov[mt.group];
    const typename XBuf<XT>::ptr x = XBuf<XT>::at(ws, mt.x0, mt);
    const int nv = ch.len >> 2;
    float ss = 0.f;
    if (ch.vec) {
      const float* g = G.p[ch.shard] + ch.shard_off;
      float* m = M.p[ch.shard] + ch.shard_off;
      const typename XBuf<XT>::ptr xv = x + ch.local;
      const float4* g4 = reinterpret_cast<const float4*>(g);
      float4* m4 = reinterpret_cast<float4*>(m);
      int v = threadIdx.x;
      for (; v + 3 * kThreads < nv; v += 4 * kThreads) {
        float4 gv[4], mv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          gv[u] = __ldcs(g4 + v + u * kThreads);
          mv[u] = __ldcs(m4 + v + u * kThreads);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          float4 mn, xn;
          mn.x = fmaf(mu, mv[u].x, gv[u].x);
          mn.y = fmaf(mu, mv[u].y, gv[u].y);
          mn.z = fmaf(mu, mv[u].z, gv[u].z);
          mn.w = fmaf(mu, mv[u].w, gv[u].w);
          if (nesterov) {
            xn.x = fmaf(mu, mn.x, gv[u].x);
            xn.y = fmaf(mu, mn.y, gv[u].y);
            xn.z = fmaf(mu, mn.z, gv[u].z);
            xn.w = fmaf(mu, mn.w, gv[u].w);
          } else {
            xn = mn;
          }
          __stcs(m4 + v + u * kThreads, mn);
          store4(xv + 4 * (v + u * kThreads), xn.x, xn.y, xn.z, xn.w);
          ss = add_sq4(ss, xn.x, xn.y, xn.z, xn.w);
        }
      }
      for (; v < nv; v += kThreads) {
        const float4 gv = __ldcs(g4 + v);
        const float4 mv = __ldcs(m4 + v);
        float4 mn, xn;
        mn.x = fmaf(mu, mv.x, gv.x);
        mn.y = fmaf(mu, mv.y, gv.y);
        mn.z = fmaf(mu, mv.z, gv.z);
        mn.w = fmaf(mu, mv.w, gv.w);
        if (nesterov) {
          xn.x = fmaf(mu, mn.x, gv.x);
          xn.y = fmaf(mu, mn.y, gv.y);
          xn.z = fmaf(mu, mn.z, gv.z);
          xn.w = fmaf(mu, mn.w, gv.w);
        } else {
          xn = mn;
        }
        __stcs(m4 + v, mn);
        store4(xv + 4 * v, xn.x, xn.y, xn.z, xn.w);
        ss = add_sq4(ss, xn.x, xn.y, xn.z, xn.w);
      }
      for (int t = nv * 4 + threadIdx.x; t < ch.len; t += kThreads) {
        const float mn = fmaf(mu, m[t], g[t]);
        const float xn = nesterov ? fmaf(mu, mn, g[t]) : mn;
        m[t] = mn;
        store1(xv + t, xn);
        ss = add_sq1(ss, xn);
      }
    } else {
      // Same element-to-thread assignment and summation order as the 128-bit path.
      for (int v = threadIdx.x; v < nv; v += kThreads) {
        float xs[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int t = 4 * v + e;
          const float gt = *elem_ptr(G, ch, L, t);
          float* mp = elem_ptr(M, ch, L, t);
          const float mn = fmaf(mu, *mp, gt);
          const float xn = nesterov ? fmaf(mu, mn, gt) : mn;
          *mp = mn;
          store1(x + x_index(mt, ch.local + t), xn);
          xs[e] = xn;
        }
        ss = add_sq4(ss, xs[0], xs[1], xs[2], xs[3]);
      }
      for (int t = nv * 4 + threadIdx.x; t < ch.len; t += kThreads) {
        const float gt = *elem_ptr(G, ch, L, t);
        float* mp = elem_ptr(M, ch, L, t);
        const float mn = fmaf(mu, *mp, gt);
        const float xn = nesterov ? fmaf(mu, mn, gt) : mn;
        *mp = mn;
        store1(x + x_index(mt, ch.local + t), xn);
        ss = add_sq1(ss, xn);
      }
    }
    const float tot = block_sum(ss, red);
    if (threadIdx.x == 0) partials[ci] = tot;
  }
}

template <typename XT>
__global__ void __launch_bounds__(kThreads)
full_input_kernel(const ChunkDev* __restrict__ chunks, int64_t n_chunks,
                  const MatDev* __restrict__ mats, const float* __restrict__ full,
                  uint8_t* __restrict__ ws, float* __restrict__ partials, const DebugCtx dbg) {
  __shared__ float red[32];
  if (debug_halted(dbg)) return;
  for (int64_t ci = blockIdx.x; ci < n_chunks; ci += gridDim.x) {
    const ChunkDev ch = chunks[ci];
    if (kDebugChecks && !debug_chunk_ok(ch, mats, dbg, nullptr)) continue;
    const MatDev& mt = mats[ch.mat];
    const float* src = full + mt.full_off + ch.local;
    const typename XBuf<XT>::ptr x = XBuf<XT>::at(ws, mt.x0, mt);
    float ss = 0.f;
    for (int t = threadIdx.x; t < ch.len; t += kThreads) {
      const float v = src[t];
      store1(x + x_index(mt, ch.local + t), v);
      ss = add_sq1(ss, v);
    }
    const float tot = block_sum(ss, red);
    if (threadIdx.x == 0) partials[ci] = tot;
  }
}

__global__ void __launch_bounds__(kThreads)
norm_finalize_kernel(const MatDev* __restrict__ mats, int n_mats,
                     const float* __restrict__ partials, float* __restrict__ inv_norm,
                     int64_t n_chunks, const DebugCtx dbg) {
  __shared__ double red[kThreads];
  if (debug_halted(dbg)) return;
  for (int mi = blockIdx.x; mi < n_mats; mi += gridDim.x) {
    const MatDev& mt = mats[mi];
    if (kDebugChecks && (mt.chunk_begin < 0 || mt.chunk_end > n_chunks ||
                         mt.chunk_begin > mt.chunk_end)) {
      if (threadIdx.x == 0) debug_fail(dbg);
      continue;
    }
    double s = 0.0;
    for (int64_t c = mt.chunk_begin + threadIdx.x; c < mt.chunk_end; c += kThreads)
      s += (double)partials[c];
    red[threadIdx.x] = s;
    __syncthreads();
    for (int w = kThreads / 2; w > 0; w >>= 1) {
      if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
      __syncthreads();
    }
    if (threadIdx.x == 0) inv_norm[mi] = red[0] > 0.0 ? (float)(1.0 / sqrt(red[0])) : 0.f;
    __syncthreads();
  }
}

template <typename XT>
__global__ void __launch_bounds__(kThreads)
apply_kernel(const ChunkDev* __restrict__ chunks, int64_t n_chunks,
             const MatDev* __restrict__ mats, ShardPtrs W, int64_t L,
             const uint8_t* __restrict__ ws,
             int final_buf, const float* __restrict__ inv_norm, int pending_norm,
             const __grid_constant__ GroupParams gp, const DebugCtx dbg) {
  if (debug_halted(dbg)) return;
  for (int64_t ci = blockIdx.x; ci < n_chunks; ci += gridDim.x) {
    const ChunkDev ch = chunks[ci];
    if (kDebugChecks && !debug_chunk_ok(ch, mats, dbg, &W)) continue;
    const MatDev& mt = mats[ch.mat];
    float lrs = gp.lr[mt.group] * mt.scale;
    const float decay = gp.decay[mt.group];
    if (pending_norm) lrs *= inv_norm[ch.mat];
    const typename XBuf<XT>::ptr o = XBuf<XT>::at(ws, final_buf ? mt.x1 : mt.x0, mt);
    if (ch.vec) {
      float* __restrict__ w = W.p[ch.shard] + ch.shard_off;
      const typename XBuf<XT>::ptr ov = o + ch.local;
      float4* w4 = reinterpret_cast<float4*>(w);
      const int nv = ch.len >> 2;
      int v = threadIdx.x;
      for (; v + 3 * kThreads < nv; v += 4 * kThreads) {
        float4 wv[4], of[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          wv[u] = __ldcs(w4 + v + u * kThreads);
          of[u] = load4(ov + 4 * (v + u * kThreads));
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          float4 r;
          r.x = fmaf(-lrs, of[u].x, wv[u].x * decay);
          r.y = fmaf(-lrs, of[u].y, wv[u].y * decay);
          r.z = fmaf(-lrs, of[u].z, wv[u].z * decay);
          r.w = fmaf(-lrs, of[u].w, wv[u].w * decay);
          __stcs(w4 + v + u * kThreads, r);
        }
      }
      for (; v < nv; v += kThreads) {
        const float4 wv = __ldcs(w4 + v);
        const float4 of = load4(ov + 4 * v);
        float4 r;
        r.x = fmaf(-lrs, of.x, wv.x * decay);
        r.y = fmaf(-lrs, of.y, wv.y * decay);
        r.z = fmaf(-lrs, of.z, wv.z * decay);
        r.w = fmaf(-lrs, of.w, wv.w * decay);
        __stcs(w4 + v, r);
      }
      for (int t = nv * 4 + threadIdx.x; t < ch.len; t += kThreads)
        w[t] = fmaf(-lrs, load1(ov + t), w[t] * decay);
    } else {
      for (int t = threadIdx.x; t < ch.len; t += kThreads) {
        float* wp = elem_ptr(W, ch, L, t);
        *wp = fmaf(-lrs, load1(o + x_index(mt, ch.local + t)), *wp * decay);
      }
    }
  }
}

__global__ void __launch_bounds__(kThreads)
gather_kernel(const ChunkDev* __restrict__ chunks, int64_t n_chunks,
              const MatDev* __restrict__ mats, ShardPtrs S, int64_t L, float* __restrict__ full,
              const DebugCtx dbg) {
  if (debug_halted(dbg)) return;
  for (int64_t ci = blockIdx.x; ci < n_chunks; ci += gridDim.x) {
    const ChunkDev ch = chunks[ci];
    if (kDebugChecks && !debug_chunk_ok(ch, mats, dbg, &S)) continue;
    float* dst = full + mats[ch.mat].full_off + ch.local;
    if (ch.vec) {
      const float* src = S.p[ch.shard] + ch.shard_off;
      const int nv = ch.len >> 2;
      for (int v = threadIdx.x; v < nv; v += kThreads)
        reinterpret_cast<float4*>(dst)[v] = reinterpret_cast<const float4*>(src)[v];
      for (int t = nv * 4 + threadIdx.x; t < ch.len; t += kThreads) dst[t] = src[t];
    } else {
      for (int t = threadIdx.x; t < ch.len; t += kThreads) dst[t] = *elem_ptr(S, ch, L, t);
    }
  }
}

__global__ void __launch_bounds__(kThreads)
scatter_kernel(const ChunkDev* __restrict__ chunks, int64_t n_chunks,
               const MatDev* __restrict__ mats, const float* __restrict__ full, ShardPtrs D,
               int64_t L, const DebugCtx dbg) {
  if (debug_halted(dbg)) return;
  for (int64_t ci = blockIdx.x; ci < n_chunks; ci += gridDim.x) {
    const ChunkDev ch = chunks[ci];
    if (kDebugChecks && !debug_chunk_ok(ch, mats, dbg, &D)) continue;
    const float* src = full + mats[ch.mat].full_off + ch.local;
    if (ch.vec) {
      float* dst = D.p[ch.shard] + ch.shard_off;
      const int nv = ch.len >> 2;
      for (int v = threadIdx.x; v < nv; v += kThreads)
        reinterpret_cast<float4*>(dst)[v] = reinterpret_cast<const float4*>(src)[v];
      for (int t = nv * 4 + threadIdx.x; t < ch.len; t += kThreads) dst[t] = src[t];
    } else {
      for (int t = threadIdx.x; t < ch.len; t += kThreads) *elem_ptr(D, ch, L, t) = src[t];
    }
  }
}

template <typename XT>
__global__ void __launch_bounds__(kThreads)
export_kernel(const ChunkDev* __restrict__ chunks, int64_t n_chunks,
              const MatDev* __restrict__ mats, const uint8_t* __restrict__ ws, int buf,
              const float* __restrict__ inv_norm, int pending_norm, float* __restrict__ full,
              const DebugCtx dbg) {
  if (debug_halted(dbg)) return;
  for (int64_t ci = blockIdx.x; ci < n_chunks; ci += gridDim.x) {
    const ChunkDev ch = chunks[ci];
    if (kDebugChecks && !debug_chunk_ok(ch, mats, dbg, nullptr)) continue;
    const MatDev& mt = mats[ch.mat];
    const float s = pending_norm ? inv_norm[ch.mat] : 1.f;
    const typename XBuf<XT>::ptr x = XBuf<XT>::at(ws, buf ? mt.x1 : mt.x0, mt);
    float* dst = full + mt.full_off + ch.local;
    for (int t = threadIdx.x; t < ch.len; t += kThreads)
      dst[t] = load1(x + x_index(mt, ch.local + t)) * s;
  }
}

int grid_for(const Plan& plan, const DevTables& dt) {
  const int64_t n = (int64_t)plan.chunks.size();
  const int64_t cap = (int64_t)dt.n_sms * kBlocksPerSm;
  return (int)(n < cap ? n : cap);
}

}  // namespace

DebugCtx make_debug_ctx(const Plan& plan, const DevTables& dt) {
  DebugCtx d{};
  d.err = dt.err;
  d.n_mats = (int32_t)plan.mats.size();
  d.n_shards = plan.n_shards;
  d.L = plan.L > 0 ? plan.L : 1;
  d.ws_bytes = plan.ws_bytes;
  d.ns_dtype = plan.ns_dtype;
  return d;
}

cudaError_t launch_momentum_input(const Plan& plan, const DevTables& dt, const ShardPtrs& g,
                                  const ShardPtrs& m, void* ws, const GroupParams& gp,
                                  cudaStream_t st) {
  const int grid = grid_for(plan, dt);
  if (grid == 0) return cudaSuccess;
  const DebugCtx dbg = make_debug_ctx(plan, dt);
  uint8_t* w = static_cast<uint8_t*>(ws);
  float* partials = reinterpret_cast<float*>(w + plan.ws_partials);
  if (plan.ns_dtype == 0)
    momentum_input_kernel<__nv_bfloat16><<<grid, kThreads, 0, st>>>(
        dt.chunks, (int64_t)plan.chunks.size(), dt.mats, g, m, plan.L, w, partials, gp, dbg);
  else if (plan.ns_dtype == 1)
    momentum_input_kernel<float><<<grid, kThreads, 0, st>>>(
        dt.chunks, (int64_t)plan.chunks.size(), dt.mats, g, m, plan.L, w, partials, gp, dbg);
  else
    momentum_input_kernel<Bf16x3><<<grid, kThreads, 0, st>>>(
        dt.chunks, (int64_t)plan.chunks.size(), dt.mats, g, m, plan.L, w, partials, gp, dbg);
  return cudaGetLastError();
}

cudaError_t launch_full_input(const Plan& plan, const DevTables& dt, const float* full, void* ws,
                              cudaStream_t st) {
  const int grid = grid_for(plan, dt);
  if (grid == 0) return cudaSuccess;
  const DebugCtx dbg = make_debug_ctx(plan, dt);
  uint8_t* w = static_cast<uint8_t*>(ws);
  float* partials = reinterpret_cast<float*>(w + plan.ws_partials);
  if (plan.ns_dtype == 0)
    full_input_kernel<__nv_bfloat16><<<grid, kThreads, 0, st>>>(
        dt.chunks, (int64_t)plan.chunks.size(), dt.mats, full, w, partials, dbg);
  else if (plan.ns_dtype == 1)
    full_input_kernel<float><<<grid, kThreads, 0, st>>>(dt.chunks, (int64_t)plan.chunks.size(),
                                                        dt.mats, full, w, partials, dbg);
  else
    full_input_kernel<Bf16x3><<<grid, kThreads, 0, st>>>(dt.chunks, (int64_t)plan.chunks.size(),
                                                         dt.mats, full, w, partials, dbg);
  return cudaGetLastError();
}

cudaError_t launch_norm_finalize(const Plan& plan, const DevTables& dt, void* ws,
                                 cudaStream_t st) {
  const int n = (int)plan.mats.size();
  if (n == 0) return cudaSuccess;
  uint8_t* w = static_cast<uint8_t*>(ws);
  const int grid = n < 65535 ? n : 65535;
  norm_finalize_kernel<<<grid, kThreads, 0, st>>>(
      dt.mats, n, reinterpret_cast<const float*>(w + plan.ws_partials),
      reinterpret_cast<float*>(w + plan.ws_inv_norm), (int64_t)plan.chunks.size(),
      make_debug_ctx(plan, dt));
  return cudaGetLastError();
}

cudaError_t launch_apply(const Plan& plan, const DevTables& dt, const ShardPtrs& wp,
                         const void* ws, int final_buf, int pending_norm, const GroupParams& gp,
                         cudaStream_t st) {
  const int grid = grid_for(plan, dt);
  if (grid == 0) return cudaSuccess;
  const DebugCtx dbg = make_debug_ctx(plan, dt);
  const uint8_t* w = static_cast<const uint8_t*>(ws);
  const float* inv = reinterpret_cast<const float*>(w + plan.ws_inv_norm);
  if (plan.ns_dtype == 0)
    apply_kernel<__nv_bfloat16><<<grid, kThreads, 0, st>>>(
        dt.chunks, (int64_t)plan.chunks.size(), dt.mats, wp, plan.L, w, final_buf, inv,
        pending_norm, gp, dbg);
  else if (plan.ns_dtype == 1)
    apply_kernel<float><<<grid, kThreads, 0, st>>>(dt.chunks, (int64_t)plan.chunks.size(),
                                                   dt.mats, wp, plan.L, w, final_buf, inv,
                                                   pending_norm, gp, dbg);
  else
    apply_kernel<Bf16x3><<<grid, kThreads, 0, st>>>(dt.chunks, (int64_t)plan.chunks.size(),
                                                    dt.mats, wp, plan.L, w, final_buf, inv,
                                                    pending_norm, gp, dbg);
  return cudaGetLastError();
}

cudaError_t launch_gather(const Plan& plan, const DevTables& dt, const ShardPtrs& src,
                          float* full, cudaStream_t st) {
  const int grid = grid_for(plan, dt);
  if (grid == 0) return cudaSuccess;
  gather_kernel<<<grid, kThreads, 0, st>>>(dt.chunks, (int64_t)plan.chunks.size(), dt.mats,
                                           src, plan.L, full, make_debug_ctx(plan, dt));
  return cudaGetLastError();
}

cudaError_t launch_scatter(const Plan& plan, const DevTables& dt, const float* full,
                           const ShardPtrs& dst, cudaStream_t st) {
  const int grid = grid_for(plan, dt);
  if (grid == 0) return cudaSuccess;
  scatter_kernel<<<grid, kThreads, 0, st>>>(dt.chunks, (int64_t)plan.chunks.size(), dt.mats,
                                            full, dst, plan.L, make_debug_ctx(plan, dt));
  return cudaGetLastError();
}

cudaError_t launch_export(const Plan& plan, const DevTables& dt, const void* ws, int buf,
                          int pending_norm, float* full, cudaStream_t st) {
  const int grid = grid_for(plan, dt);
  if (grid == 0) return cudaSuccess;
  const DebugCtx dbg = make_debug_ctx(plan, dt);
  const uint8_t* w = static_cast<const uint8_t*>(ws);
  const float* inv = reinterpret_cast<const float*>(w + plan.ws_inv_norm);
  if (plan.ns_dtype == 0)
    export_kernel<__nv_bfloat16><<<grid, kThreads, 0, st>>>(
        dt.chunks, (int64_t)plan.chunks.size(), dt.mats, w, buf, inv, pending_norm, full, dbg);
  else if (plan.ns_dtype == 1)
    export_kernel<float><<<grid, kThreads, 0, st>>>(dt.chunks, (int64_t)plan.chunks.size(),
                                                    dt.mats, w, buf, inv, pending_norm, full, dbg);
  else
    export_kernel<Bf16x3><<<grid, kThreads, 0, st>>>(dt.chunks, (int64_t)plan.chunks.size(),
                                                     dt.mats, w, buf, inv, pending_norm, full, dbg);
  return cudaGetLastError();
}

}  // namespace muon
