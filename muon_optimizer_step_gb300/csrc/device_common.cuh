// Device helpers shared by the kernels: bounded mbarrier waits, TMA loads, tcgen05
// (TMEM allocation, MMA, commit, loads) as inline PTX for sm_103a, bf16 packing.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "muon_internal.h"

namespace muon {

constexpr int kErrTimeout = 4;      // matches MUON_ERR_TIMEOUT
constexpr int kErrDeviceCheck = 7;  // matches MUON_ERR_DEVICE_CHECK

// Kernel arguments: up to 128 shard base pointers, passed by value.
struct ShardPtrs {
  float* p[128];
};

// ------------------------------------------------------------------ debug range checks
// A debug build (compiled with -DMUON_DEBUG) checks, inside the kernels that use them,
// every table entry before any access it drives: chunk records (matrix index, extent,
// the shard index and offset of their first and last element, non-null shard pointers),
// matrix records (shape, pitches, workspace buffers inside the workspace, flat extent
// inside the shards) and tile records (matrix index, tile origin on the tile grid and
// inside the phase's output, reduction length).  A failed check records
// MUON_ERR_DEVICE_CHECK in the device error word and the kernel skips the work the entry
// drives (or, for the pipelined tensor-core kernels, the whole launch); kernels that
// start after a failed check return at once.  Nothing traps.  Release builds compile the
// checks away.
#ifdef MUON_DEBUG
constexpr bool kDebugChecks = true;
#else
constexpr bool kDebugChecks = false;
#endif

// What the checks compare against (passed to the kernels by value in every build).
struct DebugCtx {
  int* err;          // device error word
  int32_t n_mats;
  int32_t n_shards;
  int64_t L;         // shard length (elements)
  int64_t ws_bytes;  // workspace bytes
  int32_t ns_dtype;  // 0 bf16, 1 fp32, 2 split fp32
  int32_t pad_;
};

__device__ __forceinline__ bool debug_fail(const DebugCtx& d) {
  atomicExch(d.err, kErrDeviceCheck);
  return false;
}

// A failed check earlier in the stream (kept until muon_check clears it).
__device__ __forceinline__ bool debug_halted(const DebugCtx& d) {
  return kDebugChecks && *reinterpret_cast<volatile int*>(d.err) == kErrDeviceCheck;
}

__device__ __forceinline__ int64_t debug_buf_bytes(int64_t elems, int32_t ns_dtype) {
  const int64_t esz = ns_dtype == 1 ? 4 : 2;
  const int64_t parts = ns_dtype == 2 ? 3 : 1;
  const int64_t one = (elems * esz + kWsAlign - 1) / kWsAlign * kWsAlign;
  return one * parts;
}

__device__ __forceinline__ bool debug_mat_ok(const MatDev& mt, const DebugCtx& d) {
  if (mt.rows < 1 || mt.cols < 1) return false;
  if (mt.m != min(mt.rows, mt.cols) || mt.n != max(mt.rows, mt.cols)) return false;
  if (mt.tall != (mt.rows > mt.cols ? 1 : 0)) return false;
  if (mt.ldx < mt.cols || mt.lda < mt.m) return false;
  const int64_t xb = debug_buf_bytes((int64_t)mt.rows * mt.ldx, d.ns_dtype);
  const int64_t ab = debug_buf_bytes((int64_t)mt.m * mt.lda, d.ns_dtype);
  if (mt.x0 < 0 || mt.x0 + xb > d.ws_bytes || mt.x1 < 0 || mt.x1 + xb > d.ws_bytes) return false;
  if (mt.a < 0 || mt.a + ab > d.ws_bytes || mt.b < 0 || mt.b + ab > d.ws_bytes) return false;
  if ((mt.x0 | mt.x1 | mt.a | mt.b) % kWsAlign != 0) return false;
  const int64_t numel = (int64_t)mt.rows * mt.cols;
  if (mt.flat_off < 0 || mt.flat_off + numel > d.L * d.n_shards) return false;
  if (mt.group < 0 || mt.group >= kMaxGroups) return false;
  return true;
}

// Non-null shard pointers for the flat range [g0, g1) (g1 > g0).
__device__ __forceinline__ bool debug_shards_ok(const ShardPtrs& P, int64_t g0, int64_t g1,
                                                const DebugCtx& d) {
  const int64_t s0 = g0 / d.L, s1 = (g1 - 1) / d.L;
  if (s0 < 0 || s1 >= d.n_shards || s1 >= 128) return false;
  for (int64_t s = s0; s <= s1; ++s)
    if (P.p[s] == nullptr) return false;
  return true;
}

// Checks a chunk record and its matrix; P (may be null) are the shards it reads or
// writes.  Records the failure; returns whether the chunk may be used.
__device__ __forceinline__ bool debug_chunk_ok(const ChunkDev& ch, const MatDev* mats,
                                               const DebugCtx& d, const ShardPtrs* P) {
  if (ch.mat < 0 || ch.mat >= d.n_mats) return debug_fail(d);
  const MatDev& mt = mats[ch.mat];
  if (!debug_mat_ok(mt, d)) return debug_fail(d);
  const int64_t numel = (int64_t)mt.rows * mt.cols;
  if (ch.len < 1 || ch.local < 0 || ch.local + ch.len > numel) return debug_fail(d);
  const int64_t g0 = mt.flat_off + ch.local;
  if (ch.shard != g0 / d.L || ch.shard_off != g0 - (int64_t)ch.shard * d.L) return debug_fail(d);
  if (ch.vec && ch.shard_off + ch.len > d.L) return debug_fail(d);
  if (P != nullptr && !debug_shards_ok(*P, g0, g0 + ch.len, d)) return debug_fail(d);
  return true;
}

// Checks a tile record of `phase` on a bm x bn tile grid with k-blocks of bk.
__device__ __forceinline__ bool debug_tile_ok(const TileDev& t, int phase, const MatDev* mats,
                                              const DebugCtx& d, int bm, int bn, int bk) {
  if (t.mat < 0 || t.mat >= d.n_mats) return false;
  const MatDev& mt = mats[t.mat];
  if (!debug_mat_ok(mt, d)) return false;
  const int mo = phase == kPhaseUpdate ? mt.rows : mt.m;
  const int no = phase == kPhaseUpdate ? mt.cols : mt.m;
  const int K = phase == kPhaseGram ? mt.n : mt.m;
  if (t.i0 < 0 || t.i0 >= mo || t.i0 % bm != 0) return false;
  if (t.j0 < 0 || t.j0 >= no || t.j0 % bn != 0) return false;
  if (t.kblocks != (K + bk - 1) / bk) return false;
  return true;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity to complete.  Gives up after `budget`
// clock cycles (or as soon as *abort is set by another role of the block): records
// MUON_ERR_TIMEOUT in *err, sets *abort and returns false.  Never spins forever.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  long long budget, int* err,
                                                  volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (clock64() - t0 > budget) {
      atomicExch(err, kErrTimeout);
      *abort = 1;
      return false;
    }
  }
}

// ------------------------------------------------------------------ TMA
__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

__device__ __forceinline__ void tma_load_2d(void* smem_dst, const void* tmap, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem_dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// Bulk tensor store of a shared-memory box to global memory (async proxy; completion is
// tracked with bulk groups: commit, then wait_group / wait_group.read).
__device__ __forceinline__ void tma_store_2d(const void* tmap, int x, int y, uint32_t smem_src) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   tmap),
               "r"(x), "r"(y), "r"(smem_src)
               : "memory");
}

// The same store with an L2 eviction-priority hint (a createpolicy value).
__device__ __forceinline__ void tma_store_2d_hint(const void* tmap, int x, int y,
                                                  uint32_t smem_src, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group.L2::cache_hint"
      " [%0, {%1, %2}], [%3], %4;" ::"l"(tmap),
      "r"(x), "r"(y), "r"(smem_src), "l"(policy)
      : "memory");
}

// L2 policy: lines written or read under it are the first candidates for eviction.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Waits until the committed bulk stores have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Waits until the committed bulk stores have completed.
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Waits until every committed bulk-store group but the newest n has completed (n > 8
// waits for all but 8, which includes the older ones).
__device__ __forceinline__ void bulk_wait_all_but(int n) {
  switch (n) {
    case 0: asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); break;
    case 1: asm volatile("cp.async.bulk.wait_group 1;" ::: "memory"); break;
    case 2: asm volatile("cp.async.bulk.wait_group 2;" ::: "memory"); break;
    case 3: asm volatile("cp.async.bulk.wait_group 3;" ::: "memory"); break;
    case 4: asm volatile("cp.async.bulk.wait_group 4;" ::: "memory"); break;
    case 5: asm volatile("cp.async.bulk.wait_group 5;" ::: "memory"); break;
    case 6: asm volatile("cp.async.bulk.wait_group 6;" ::: "memory"); break;
    case 7: asm volatile("cp.async.bulk.wait_group 7;" ::: "memory"); break;
    default: asm volatile("cp.async.bulk.wait_group 8;" ::: "memory"); break;
  }
}

// Orders this thread's generic shared-memory writes before later async-proxy reads.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------ tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t* smem_slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(smem_slot)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16 (bf16 inputs, fp32 accumulator).
__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when every tcgen05.mma issued so far by this thread completes.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread t of the warp gets lane (base + t).
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor (tcgen05 format): start address, leading / stride
// byte offsets, fixed 0b001 at bits 46-48, swizzle mode at bits 61-63 (2 = 128-byte).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo,
                                                    uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFF) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B, operand majors
// (0 = K-major, 1 = MN-major), N >> 3 at bits 17-22, M >> 4 at bits 24-28.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int a_mn, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) |
         ((uint32_t)b_mn << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// ------------------------------------------------------------------ split fp32 (bf16 x 3)
// An fp32 value x kept as three bf16 values h = bf16(x), m = bf16(x - h),
// l = bf16(x - h - m) (each difference is exact in fp32), in three equal arrays: the m
// and l arrays of a buffer follow its h array, each sized to whole kWsAlign units.
// h + m + l recovers x to within 2^-26 |x|, and a product of two such values is
// hh + hm + mh + hl + lh + mm up to about 2^-26 of it (the ml, lm, ll terms are dropped),
// below the rounding of one fp32 product.
struct Bf16x3 {};

__host__ __device__ constexpr int64_t split_part_bytes(int64_t part_bytes) {
  return (part_bytes + kWsAlign - 1) / kWsAlign * kWsAlign;
}

__device__ __forceinline__ void split_bf16x3(float x, __nv_bfloat16& h, __nv_bfloat16& m,
                                             __nv_bfloat16& l) {
  h = __float2bfloat16_rn(x);
  const float r1 = x - __bfloat162float(h);
  m = __float2bfloat16_rn(r1);
  l = __float2bfloat16_rn(r1 - __bfloat162float(m));
}

// ------------------------------------------------------------------ clusters / CTA pairs
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Address of the same shared-memory offset in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}

// Arrive (with expected transaction bytes) on an mbarrier that may live in the peer CTA.
__device__ __forceinline__ void mbar_arrive_expect_tx_cluster(uint32_t cluster_addr, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cluster.shared::cluster.b64 _, [%0], %1;"
               ::"r"(cluster_addr), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

// TMA load into this CTA's shared memory that signals an mbarrier in either CTA of the pair.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t smem_dst, const void* tmap, int x, int y,
                                                 uint32_t bar_cluster_addr) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_dst),
      "l"(tmap), "r"(x), "r"(y), "r"(bar_cluster_addr)
      : "memory");
}

__device__ __forceinline__ void tmem_alloc_pair(uint32_t* smem_slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(smem_slot)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// D[tmem of both CTAs] (+)= A[smem of both] * B[smem of both]^T, issued by the even CTA.
__device__ __forceinline__ void tc_mma_f16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on the barrier at this offset in every CTA of `mask` when the pair's
// previously issued MMAs complete.
__device__ __forceinline__ void tc_commit_pair(uint64_t* bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(smem_u32(bar)), "h"(mask)
      : "memory");
}

// ------------------------------------------------------------------ fused apply
// Per-group hyper-parameters of one call (group g of a matrix = MatDev::group).
struct GroupParams {
  float lr[kMaxGroups];
  float decay[kMaxGroups];  // 1 - lr * wd
  float mu[kMaxGroups];
  int nesterov[kMaxGroups];
};

// Arguments of the last Newton-Schulz Update when it also applies the step to the weights.
struct ApplyArgs {
  ShardPtrs W;     // parameter shards
  long long L;     // shard length
  float inv_L;     // 1 / L, rounded to fp32 (shard_of's estimate)
  GroupParams gp;  // lr and decay per group
};

// Shard and in-shard offset of flat element g (0 <= g < n_shards * L), without a 64-bit
// division: the fp32 estimate of g / L (< 2^7) is off by at most one, and is corrected.
__device__ __forceinline__ long long shard_of(const ApplyArgs& ap, long long g, long long* off) {
  long long s = (long long)((float)g * ap.inv_L);
  long long o = g - s * ap.L;
  if (o < 0) {
    --s;
    o += ap.L;
  } else if (o >= ap.L) {
    ++s;
    o -= ap.L;
  }
  *off = o;
  return s;
}

// Debug builds: the shards a matrix's apply writes exist.
__device__ __forceinline__ bool debug_apply_ok(const ApplyArgs& ap, const MatDev& mt,
                                               const DebugCtx& d) {
  return debug_shards_ok(ap.W, mt.flat_off, mt.flat_off + (int64_t)mt.rows * mt.cols, d);
}

// W <- W * decay - lr * scale * O for the elements (i, jb .. jb + n - 1) of a matrix, whose
// row-major element (i, j) lives at flat index flat_off + i * cols + j of the sharded
// buffer.  o holds the fp32 update values.  128-bit accesses when the run lies in one
// shard and is aligned, element by element otherwise.
__device__ __forceinline__ void apply_row_run(const ApplyArgs& ap, const MatDev& mt, int i, int jb,
                                              int n, const float (&o)[32]) {
  const float lrs = ap.gp.lr[mt.group] * mt.scale;
  const float decay = ap.gp.decay[mt.group];
  const long long g0 = mt.flat_off + (long long)i * mt.cols + jb;
  long long off0;
  const long long s0 = shard_of(ap, g0, &off0);
  if (n == 32 && off0 + 32 <= ap.L && (off0 & 3) == 0) {
    float4* w = reinterpret_cast<float4*>(ap.W.p[s0] + off0);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      float4 v = __ldcs(w + q);
      v.x = fmaf(-lrs, o[4 * q + 0], v.x * decay);
      v.y = fmaf(-lrs, o[4 * q + 1], v.y * decay);
      v.z = fmaf(-lrs, o[4 * q + 2], v.z * decay);
      v.w = fmaf(-lrs, o[4 * q + 3], v.w * decay);
      __stcs(w + q, v);
    }
  } else {
#pragma unroll
    for (int t = 0; t < 32; ++t) {
      if (t < n) {
        long long off;
        const long long s = shard_of(ap, g0 + t, &off);
        float* w = ap.W.p[s] + off;
        *w = fmaf(-lrs, o[t], *w * decay);
      }
    }
  }
}

// Asks L2 to fetch n weights of matrix row i from column jb: one bulk prefetch when the
// run lies in one shard and starts on a 16-byte boundary (shard bases are 16-byte
// aligned), nothing otherwise.  A hint: no data reaches the SM and nothing waits on it.
__device__ __forceinline__ void prefetch_w_row(const ApplyArgs& ap, const MatDev& mt, int i,
                                               int jb, int n) {
  if (i >= mt.rows || jb >= mt.cols) return;
  n = min(n, mt.cols - jb);
  const long long g0 = mt.flat_off + (long long)i * mt.cols + jb;
  long long off;
  const long long s = shard_of(ap, g0, &off);
  const uint32_t bytes = (uint32_t)(4 * n) & ~15u;
  if (bytes == 0 || off + n > ap.L || (off & 3) != 0) return;
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(ap.W.p[s] + off), "r"(bytes)
               : "memory");
}

// W <- W*decay - lr*scale*O on the 32 x 32 block of matrix mt at rows r0.., columns jb..,
// whose fp32 O the warp holds one row per lane (o = row r0 + lane).  The lanes' rows are
// 4 KB apart in W, so the block is first turned around in `scratch` (4 KB of shared
// memory, 16-byte aligned, not read by any pending bulk store): 16-byte chunk k of row r
// goes to slot 8r + (k ^ (r & 7)), which keeps both passes free of bank conflicts.  Each
// weight access then covers four whole rows (8 lanes x 16 bytes per row), and the eight
// loads of a lane are all issued before the first store.  Chunks past the matrix are
// skipped; a chunk that leaves its shard or a 16-byte boundary goes element by element.
__device__ __forceinline__ void apply_block(const ApplyArgs& ap, const MatDev& mt, int r0, int jb,
                                            int lane, const float (&o)[32], uint8_t* scratch) {
  float4* sc = reinterpret_cast<float4*>(scratch);
#pragma unroll
  for (int k = 0; k < 8; ++k)
    sc[8 * lane + (k ^ (lane & 7))] = make_float4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
  __syncwarp();
  const float lrs = ap.gp.lr[mt.group] * mt.scale;
  const float decay = ap.gp.decay[mt.group];
  const int cc = lane & 7;                 // this lane's 16-byte chunk of a row
  const int col = jb + 4 * cc;
  float4 w[8];
  float* wp[8];
  bool vec[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int rr = 4 * j + (lane >> 3);    // block row of access j
    const int row = r0 + rr;
    wp[j] = nullptr;
    vec[j] = false;
    if (row < mt.rows && col < mt.cols) {
      long long off;
      const long long g = mt.flat_off + (long long)row * mt.cols + col;
      const long long sh = shard_of(ap, g, &off);
      wp[j] = ap.W.p[sh] + off;
      vec[j] = col + 4 <= mt.cols && off + 4 <= ap.L && (off & 3) == 0;
      if (vec[j]) w[j] = __ldcs(reinterpret_cast<const float4*>(wp[j]));
    }
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (wp[j] == nullptr) continue;
    const int rr = 4 * j + (lane >> 3);
    const float4 ov = sc[8 * rr + (cc ^ (rr & 7))];
    if (vec[j]) {
      float4 v = w[j];
      v.x = fmaf(-lrs, ov.x, v.x * decay);
      v.y = fmaf(-lrs, ov.y, v.y * decay);
      v.z = fmaf(-lrs, ov.z, v.z * decay);
      v.w = fmaf(-lrs, ov.w, v.w * decay);
      __stcs(reinterpret_cast<float4*>(wp[j]), v);
    } else {
      const float oe[4] = {ov.x, ov.y, ov.z, ov.w};
      const long long g = mt.flat_off + (long long)(r0 + rr) * mt.cols + col;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (col + e >= mt.cols) break;
        long long off;
        const long long sh = shard_of(ap, g + e, &off);
        float* x = ap.W.p[sh] + off;
        *x = fmaf(-lrs, oe[e], *x * decay);
      }
    }
  }
  __syncwarp();  // every lane is done with the scratch
}

// ------------------------------------------------------------------ small math helpers
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float bf16_lo(uint32_t v) {
  return __uint_as_float(v << 16);
}

__device__ __forceinline__ float bf16_hi(uint32_t v) {
  return __uint_as_float(v & 0xFFFF0000u);
}

__device__ __forceinline__ float bf16_to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

}  // namespace muon
