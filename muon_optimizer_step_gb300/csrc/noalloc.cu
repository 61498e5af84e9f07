// muon_orthogonalize_full_noalloc: Newton-Schulz of caller-given full matrices without
// any device allocation.
//
// Who needs this: a caller that cannot call cudaMalloc (or have the library call it for
// them) on the path where the orthogonalization runs.  Typical cases are a host
// framework whose caching allocator owns the device memory pool and forbids allocations
// behind its back, a latency-critical loop that cannot afford the device-wide
// synchronisation cudaMalloc / cudaFree may imply, or a plugin that runs inside a
// process where only the host application allocates device memory.  Those callers still
// pass their own input and output buffers; everything else the computation needs (the
// per-matrix work buffers X0, X1, A, B, the chunk sums of squares, 1/||X|| and the
// layout's device tables) lives in the fixed-size device array below.
#include <cstdio>
#include <cstring>
#include <string>
#include <mutex>
#include <vector>

#include "../../include/muon.h"
#include "device_common.cuh"
#include "kernels.h"
#include "layout_handle.h"

namespace {

using namespace muon;

// The scratch array of this entry point: 32 MiB on every GPU where the library's device
// code is loaded, held until the process exits.  Calls share it and leave their data in
// it; calls that overlap on the GPU (two streams, two threads) race on it.  It is
// 1024-byte aligned, so offsets that are multiples of 1024 from its start are 1024-byte
// aligned addresses, as the workspace must be.  Its first 256 bytes hold the error word
// the kernels of a debug build write (zeroed when a device is set up; muon_check reads
// and clears it).
constexpr size_t kScratchBytes = (size_t)32 << 20;
constexpr size_t kErrSlot = 256;
static __device__ __align__(1024) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDev = 64;
void* g_scratch_addr[kMaxDev] = {nullptr};
std::mutex g_scratch_mu;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Device address of the scratch array on the current device; looked up once per device
// (with that device current), when its error word is also zeroed.  The host-side name
// g_noalloc_scratch is only a stand-in.
cudaError_t scratch_address(int dev, unsigned char** out) {
  std::lock_guard<std::mutex> g(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    e = cudaMemset(p, 0, kErrSlot);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = static_cast<unsigned char*>(g_scratch_addr[dev]);
  return cudaSuccess;
}

template <typename T>
size_t place(size_t* off, size_t n, size_t align) {
  const size_t at = align_up(*off, align);
  *off = at + n * sizeof(T);
  return at;
}

}  // namespace

int* muon::noalloc_error_word(int dev) {
  if (dev < 0 || dev >= kMaxDev) return nullptr;
  std::lock_guard<std::mutex> g(g_scratch_mu);
  return static_cast<int*>(g_scratch_addr[dev]);
}

extern "C" muon_status muon_orthogonalize_full_noalloc(const muon_layout* layout,
                                                       const float* full_in, float* full_out,
                                                       int32_t ns_steps, cudaStream_t stream) {
  auto fail = [](muon_status s, const char* msg) {
    set_last_error(std::string("muon_orthogonalize_full_noalloc: ") + msg);
    return s;
  };
  if (layout == nullptr) return fail(MUON_ERR_INVALID_ARG, "layout is NULL");
  const Plan& plan = layout->plan;
  if (plan.ns_dtype != MUON_NS_FP32)
    return fail(MUON_ERR_UNSUPPORTED,
                "needs a layout created with MUON_NS_FP32 (the tensor-core path keeps TMA "
                "descriptors and a wait-status word that this entry point has no room for)");
  if (ns_steps < 0 || ns_steps > 100) return fail(MUON_ERR_INVALID_ARG, "ns_steps outside 0..100");
  if (plan.full_numel > 0) {
    if (full_in == nullptr || full_out == nullptr)
      return fail(MUON_ERR_INVALID_ARG, "full_in or full_out is NULL");
    if (reinterpret_cast<uintptr_t>(full_in) % 16 || reinterpret_cast<uintptr_t>(full_out) % 16)
      return fail(MUON_ERR_ALIGNMENT, "full_in and full_out must be 16-byte aligned");
  }
  if (plan.mats.empty()) {
    set_last_error("");
    return MUON_OK;
  }

  int dev = -1, sms = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev)
    return fail(MUON_ERR_CUDA, "no current CUDA device");
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (major != 10 || minor != 3) return fail(MUON_ERR_UNSUPPORTED, "device is not sm_103a");

  // Host-side plan of the launches (host memory only).
  TileList tl[3];
  for (int p = 0; p < 3; ++p) tl[p] = plan_tiles(plan, p, kF32BM, kF32BN, 16, sms);

  // Scratch map: the error word, the tables, then the workspace (1024-byte aligned, as
  // the kernels expect).  Everything must fit in kScratchBytes.
  size_t off = kErrSlot;
  const size_t o_chunks = place<ChunkDev>(&off, plan.chunks.size(), 256);
  const size_t o_mats = place<MatDev>(&off, plan.mats.size(), 256);
  size_t o_tiles[3], o_begin[3];
  for (int p = 0; p < 3; ++p) {
    o_tiles[p] = place<TileDev>(&off, tl[p].tiles.size(), 256);
    o_begin[p] = place<int32_t>(&off, tl[p].cta_begin.size(), 256);
  }
  const size_t o_ws = align_up(off, (size_t)kWsAlign);
  const size_t need = o_ws + (size_t)plan.ws_bytes;
  if (need > kScratchBytes) {
    char msg[320];
    std::snprintf(msg, sizeof(msg),
                  "the layout needs %zu bytes of scratch; the static scratch array holds %zu "
                  "bytes (use muon_orthogonalize_full with a caller-allocated workspace instead)",
                  need, kScratchBytes);
    return fail(MUON_ERR_UNSUPPORTED, msg);
  }

  unsigned char* base = nullptr;
  cudaError_t e = scratch_address(dev, &base);
  if (e != cudaSuccess) return fail(MUON_ERR_CUDA, cudaGetErrorString(e));

  // Upload the tables into the scratch array (pageable source: the copy is staged before
  // cudaMemcpyAsync returns, so the host vectors may go out of scope).
  auto put = [&](size_t at, const void* src, size_t bytes) -> cudaError_t {
    if (bytes == 0) return cudaSuccess;
    return cudaMemcpyAsync(base + at, src, bytes, cudaMemcpyHostToDevice, stream);
  };
  if ((e = put(o_chunks, plan.chunks.data(), plan.chunks.size() * sizeof(ChunkDev))) != cudaSuccess ||
      (e = put(o_mats, plan.mats.data(), plan.mats.size() * sizeof(MatDev))) != cudaSuccess)
    return fail(MUON_ERR_CUDA, cudaGetErrorString(e));
  DevTables dt;
  dt.device = dev;
  dt.n_sms = sms;
  dt.err = reinterpret_cast<int*>(base);
  dt.chunks = reinterpret_cast<ChunkDev*>(base + o_chunks);
  dt.mats = reinterpret_cast<MatDev*>(base + o_mats);
  for (int p = 0; p < 3; ++p) {
    if ((e = put(o_tiles[p], tl[p].tiles.data(), tl[p].tiles.size() * sizeof(TileDev))) != cudaSuccess ||
        (e = put(o_begin[p], tl[p].cta_begin.data(), tl[p].cta_begin.size() * sizeof(int32_t))) !=
            cudaSuccess)
      return fail(MUON_ERR_CUDA, cudaGetErrorString(e));
    dt.tiles[p] = reinterpret_cast<TileDev*>(base + o_tiles[p]);
    dt.cta_begin[p] = reinterpret_cast<int32_t*>(base + o_begin[p]);
    dt.grid[p] = tl[p].grid;
    dt.n_tiles[p] = (int64_t)tl[p].tiles.size();
  }
  // Nothing in the workspace has to start at zero: every slot a kernel reads (chunk sums,
  // 1/||X||, X0, X1, A, B) is written earlier in the same call.
  void* ws = base + o_ws;
  if (reinterpret_cast<uintptr_t>(ws) % kWsAlign != 0)
    return fail(MUON_ERR_ALIGNMENT, "scratch workspace is not 1024-byte aligned");
  if ((e = launch_full_input(plan, dt, full_in, ws, stream)) != cudaSuccess ||
      (e = launch_norm_finalize(plan, dt, ws, stream)) != cudaSuccess)
    return fail(MUON_ERR_CUDA, cudaGetErrorString(e));
  for (int it = 0; it < ns_steps; ++it)
    for (int ph = 0; ph < 3; ++ph)
      if ((e = launch_ns_phase_f32(plan, dt, ws, ph, it & 1, it == 0 ? 1 : 0, stream)) != cudaSuccess)
        return fail(MUON_ERR_CUDA, cudaGetErrorString(e));
  if ((e = launch_export(plan, dt, ws, ns_steps & 1, ns_steps == 0 ? 1 : 0, full_out, stream)) !=
      cudaSuccess)
    return fail(MUON_ERR_CUDA, cudaGetErrorString(e));
  set_last_error("");
  return MUON_OK;
}
