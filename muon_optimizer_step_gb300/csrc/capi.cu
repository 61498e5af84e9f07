// C ABI of libmuon.so: argument validation, device tables, and the launch sequence of the
// Muon step.  The step follows FsdpMuon._step_group of the Megatron-Core API docs
// ("core.distributed.fsdp.src.megatron_fsdp.experimental.muon"): its three stages
// (momentum inputs, orthogonalization on the owner, local apply) run for one flat
// buffer per call, enqueued on the stream the caller passes.  With one GPU the owner is this device and the gather /
// scatter of "Add initial Muon+M-FSDPv2 implementation" ("Opt step" steps 3 and 5) are
// index maps fused into the first and last kernels.
#include <cmath>
#include <cstdarg>
#include <algorithm>
#include <cstdint>
#include <cstdlib>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/muon.h"
#include "device_common.cuh"
#include "kernels.h"

using namespace muon;

#include "layout_handle.h"

namespace {

thread_local std::string g_last_error;
constexpr long long kDefaultBudget = 4000000000LL;  // ~2 s of SM clock per wait
// Newton-Schulz work of one iteration (flops, symmetric count) from which a buffer counts
// as a long step that runs at the power limit, and the tile shape such buffers get.
constexpr double kLongStepFlops = 20e12;
constexpr int kLongStepShape = kShapeSingle;
// Newton-Schulz work of one iteration below which a buffer runs as one persistent launch.
constexpr double kPersistentFlops = 1e12;
// Iterations with their own tile lists in a persistent launch (later ones reuse the last).
constexpr int kPersistentIters = 6;
// Flop-weighted mean of m (the reduction length of Poly and Update) from which a buffer
// below the long-step cut runs 256 x 512 CTA-pair tiles.
constexpr double kWideTileMeanM = 3072.0;
constexpr int kMaxDevices = 64;
int* g_err_word[kMaxDevices] = {nullptr};
std::mutex g_err_mu;

muon_status fail(muon_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

muon_status ok() {
  g_last_error.clear();
  return MUON_OK;
}

muon_status cuda_fail(cudaError_t e, const char* what) {
  return fail(MUON_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Device word where kernels record a wait that ran out (one per device, zeroed).
muon_status err_word(int dev, int** out) {
  if (dev < 0 || dev >= kMaxDevices) return fail(MUON_ERR_UNSUPPORTED, "device %d out of range", dev);
  std::lock_guard<std::mutex> g(g_err_mu);
  if (g_err_word[dev] == nullptr) {
    int* p = nullptr;
    cudaError_t e = cudaMalloc(&p, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(error word)");
    e = cudaMemset(p, 0, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemset(error word)");
    g_err_word[dev] = p;
  }
  *out = g_err_word[dev];
  return MUON_OK;
}

template <typename T>
muon_status upload(const std::vector<T>& v, T** dst) {
  *dst = nullptr;
  if (v.empty()) return MUON_OK;
  cudaError_t e = cudaMalloc(dst, v.size() * sizeof(T));
  if (e != cudaSuccess) return fail(MUON_ERR_OOM, "cudaMalloc(%zu B) for a layout table: %s",
                                    v.size() * sizeof(T), cudaGetErrorString(e));
  e = cudaMemcpy(*dst, v.data(), v.size() * sizeof(T), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(layout table)");
  return MUON_OK;
}

void free_tables(DevTables* dt) {
  if (dt->device < 0) return;
  int cur = -1;
  cudaGetDevice(&cur);
  if (cur != dt->device) cudaSetDevice(dt->device);
  cudaFree(dt->chunks);
  cudaFree(dt->mats);
  for (int p = 0; p < 3; ++p) {
    cudaFree(dt->tiles[p]);
    cudaFree(dt->cta_begin[p]);
  }
  cudaFree(dt->tc_tiles);
  cudaFree(dt->tc_begin);
  cudaFree(dt->tmaps);
  if (cur >= 0 && cur != dt->device) cudaSetDevice(cur);
  *dt = DevTables{};
}

// Uploads the layout's tables to the current device on first use.
muon_status ensure_device(muon_layout* L) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  DevTables& dt = L->dt;
  if (dt.device >= 0) {
    if (dt.device != dev)
      return fail(MUON_ERR_UNSUPPORTED, "layout was prepared on device %d, current device is %d",
                  dt.device, dev);
    return MUON_OK;
  }
  int major = 0, minor = 0, sms = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (major != 10 || minor != 3)
    return fail(MUON_ERR_UNSUPPORTED, "libmuon is built for sm_103a; device %d is sm_%d%d", dev,
                major, minor);
  DevTables t;
  t.device = dev;
  t.n_sms = sms;
  muon_status s;
  if ((s = err_word(dev, &t.err)) != MUON_OK) return s;
  if ((s = upload(L->plan.chunks, &t.chunks)) != MUON_OK) { free_tables(&t); return s; }
  const bool tc = L->plan.ns_dtype != MUON_NS_FP32;  // a tcgen05 path (bf16 or split fp32)
  const bool split = L->plan.ns_dtype == MUON_NS_SPLIT_FP32;
  if (!tc) {
    for (int p = 0; p < 3; ++p) {
      const TileList tl = plan_tiles(L->plan, p, kF32BM, kF32BN, 16, sms);
      t.grid[p] = tl.grid;
      t.n_tiles[p] = (int64_t)tl.tiles.size();
      if ((s = upload(tl.tiles, &t.tiles[p])) != MUON_OK) { free_tables(&t); return s; }
      if ((s = upload(tl.cta_begin, &t.cta_begin[p])) != MUON_OK) { free_tables(&t); return s; }
    }
  } else if (!L->plan.mats.empty()) {
    int pairs = 0, singles = 0;
    e = prepare_ns_kernels(&pairs, &singles);
    if (e != cudaSuccess) { free_tables(&t); return cuda_fail(e, "prepare tcgen05 kernels"); }
    pairs = std::min(pairs, sms / 2);
    singles = std::min(singles, sms);
    if (singles < 1) {
      free_tables(&t);
      return fail(MUON_ERR_UNSUPPORTED, "the tcgen05 kernel does not fit on an SM of device %d", dev);
    }
    // Three tile shapes, measured on GB300 (bench, bf16, alternating runs in one call):
    //  - Steps long enough to hold the GPU at its 1.4 kW limit (the 32-layer Llama-3-8B
    //    set) are decided by energy per flop: single CTAs hold the highest clock and
    //    finish first (346 ms against 351 for 256 x 512 pair tiles and 353 for pairs).
    //  - Below the limit the tensor work per clock decides.  With long reductions (two
    //    Llama layers: flop-weighted mean m of 4000) 256 x 512 pair tiles, with half the
    //    operand bytes per flop of single CTAs, win: 19.24 against 20.2 ms for pairs and
    //    20.9 for single CTAs.  With short ones (MoE: m = 1408; GPT-2: m = 768) their
    //    unoverlapped epilogue costs more than that saves (MoE 16.6 against 14.8 ms), and
    //    pairs or single CTAs tie.
    // The cut between the regimes is the Newton-Schulz work of one iteration (94 TFLOP on
    // the 32-layer set, 6 on the two-layer one) and the flop-weighted mean of m.
    double all = 0.0, m_sum = 0.0;  // one iteration's flops (3 m^2 n + m^3 per matrix)
    for (const MatDev& m : L->plan.mats) {
      const double f = 3.0 * m.m * (double)m.m * m.n + (double)m.m * m.m * m.m;
      all += f;
      m_sum += f * m.m;
    }
    const double mean_m = all > 0.0 ? m_sum / all : 0.0;
    int shape = pairs < 1 ? kShapeSingle
              : all >= kLongStepFlops ? kLongStepShape
              : mean_m >= kWideTileMeanM ? kShapePairWide : kShapePair;
    const char* v = split ? nullptr : std::getenv("MUON_TC_KERNEL");  // "1"-"3" pins a shape
    if (split) {
      // The split-fp32 kernel exists for CTA pairs only (two 96 KB operand stages).
      if (pairs < 1) {
        free_tables(&t);
        return fail(MUON_ERR_UNSUPPORTED,
                    "the split-fp32 kernel needs 2-CTA clusters, and none fits on device %d", dev);
      }
      shape = kShapePair;
    }
    if (v != nullptr && v[0] != '\0') {
      if (v[0] < '1' || v[0] > '3' || v[1] != '\0') {
        free_tables(&t);
        return fail(MUON_ERR_INVALID_ARG, "MUON_TC_KERNEL=%s: the tile shapes are 1 (single "
                    "CTA), 2 (CTA pair) and 3 (CTA pair, 256 x 512 tiles)", v);
      }
      shape = v[0] - '0';
      if (shape != kShapeSingle && pairs < 1) {
        free_tables(&t);
        return fail(MUON_ERR_UNSUPPORTED,
                    "MUON_TC_KERNEL=%d asks for 2-CTA clusters, but none of the tcgen05 "
                    "kernel fits on device %d", shape, dev);
      }
    }
    const bool cluster = shape != kShapeSingle;
    t.tc_shape = shape;
    t.tc_units = cluster ? pairs : singles;
    // One launch per phase, each phase's tiles balanced on their own, except for tiny
    // buffers: there fixed costs per launch weigh most, and the persistent launch (every
    // phase in one launch, tiles waiting on per-matrix counters) measured faster on
    // GPT-2-small with CTA pairs (1.487 against 1.572 ms per step, before its tile lists
    // were planned from a simulated run; 1.409 after) but slower on MoE (15.4 against
    // 14.8 ms) and two Llama layers (20.9 against 19.2 ms), planned lists included.  The split-fp32
    // epilogue writes with plain stores, which the persistent launch's counters do not
    // publish to the next phase's TMA reads, so it never runs persistent.
    t.tc_persistent = !split && all < kPersistentFlops;
    const char* pv = split ? nullptr : std::getenv("MUON_NS_PERSISTENT");  // "1"/"0" pins it
    if (pv != nullptr && (pv[0] == '0' || pv[0] == '1')) t.tc_persistent = pv[0] == '1';
    // Where the update is applied to W.  On long steps the last Update's epilogue does it
    // (fused tail): its reductions are long, so the weight traffic hides under the MMAs
    // and one pass over W and O is saved (Llama-3-8B set: 6-7 ms of a 359 ms step).  Short
    // reductions make the epilogue the bottleneck, and there the streaming apply kernel
    // after the last Update is cheaper (GPT-2-small: the fused tail cost 470 us of a
    // 2.06 ms step, a separate pass over W and O about 130 us).
    t.fused_tail = all >= kLongStepFlops;
    const char* fv = std::getenv("MUON_FUSED_TAIL");  // "1"/"0" pins it
    if (fv != nullptr && (fv[0] == '0' || fv[0] == '1')) t.fused_tail = fv[0] == '1';
    for (MatDev& m : L->plan.mats) m.sig[0] = m.sig[1] = m.sig[2] = 0;
    const int bm = cluster ? 256 : kTcBM;
    const int bn = shape == kShapePairWide ? 512 : cluster ? 256 : kTcBN;
    std::vector<TileList> lists;
    if (t.tc_persistent) {
      // Lists per iteration: matrices reach each phase at different times, so the best
      // order of a phase's tiles differs from one iteration to the next.
      lists = plan_persistent(L->plan, bm, bn, kTcBK, t.tc_units, kPersistentIters);
    } else {
      for (int p = 0; p < 3; ++p) lists.push_back(plan_tiles(L->plan, p, bm, bn, kTcBK, t.tc_units));
    }
    for (int p = 0; p < 3; ++p)
      for (const TileDev& td : lists[p].tiles) L->plan.mats[td.mat].sig[p] += cluster ? 2 : 1;
    // Back to back; every unit of a launch reads begin[unit + 1], so each list's offsets
    // are padded to tc_units + 1 entries.
    std::vector<TileDev> all_tiles;
    std::vector<int32_t> all_begin;
    for (TileList& tl : lists) {
      while ((int)tl.cta_begin.size() < t.tc_units + 1) tl.cta_begin.push_back(tl.cta_begin.back());
      for (int u = 0; u <= t.tc_units; ++u)
        all_begin.push_back((int32_t)all_tiles.size() + tl.cta_begin[u]);
      all_tiles.insert(all_tiles.end(), tl.tiles.begin(), tl.tiles.end());
    }
    if (all_tiles.size() > (size_t)INT32_MAX) {
      free_tables(&t);
      return fail(MUON_ERR_UNSUPPORTED, "more than 2^31 Newton-Schulz tiles");
    }
    t.tc_lists = (int)lists.size();
    t.tc_n_tiles = (int64_t)all_tiles.size();
    if ((s = upload(all_tiles, &t.tc_tiles)) != MUON_OK) { free_tables(&t); return s; }
    if ((s = upload(all_begin, &t.tc_begin)) != MUON_OK) { free_tables(&t); return s; }
    e = cudaMalloc(&t.tmaps, L->plan.mats.size() * kMapsPerMat * sizeof(CUtensorMap));
    if (e != cudaSuccess) { free_tables(&t); return fail(MUON_ERR_OOM, "cudaMalloc(tensor maps)"); }
  }
  if ((s = upload(L->plan.mats, &t.mats)) != MUON_OK) { free_tables(&t); return s; }
  dt = t;
  return MUON_OK;
}

// Encodes the TMA descriptors for this workspace (tensor-core paths) when it changes.
muon_status ensure_tmaps(muon_layout* L, const void* ws) {
  DevTables& dt = L->dt;
  if (L->plan.ns_dtype == MUON_NS_FP32 || L->plan.mats.empty() || dt.tmap_ws == ws)
    return MUON_OK;
  std::vector<CUtensorMap> maps;
  std::string err;
  if (!encode_tensor_maps(L->plan, ws, &maps, &err)) return fail(MUON_ERR_CUDA, "%s", err.c_str());
  // Kernels launched with the previous descriptors may still run on other streams.
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  e = cudaMemcpy(dt.tmaps, maps.data(), maps.size() * sizeof(CUtensorMap), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(tensor maps)");
  dt.tmap_ws = ws;
  return MUON_OK;
}

muon_status check_shards(const muon_layout* L, const void* const* shards, const char* name,
                         ShardPtrs* out) {
  std::memset(out, 0, sizeof(*out));
  if (shards == nullptr) return fail(MUON_ERR_INVALID_ARG, "%s is NULL", name);
  for (int s = 0; s < L->plan.n_shards; ++s) {
    const void* p = shards[s];
    if (p == nullptr) {
      if (L->plan.L > 0) return fail(MUON_ERR_INVALID_ARG, "%s[%d] is NULL", name, s);
    } else if (reinterpret_cast<uintptr_t>(p) % 16 != 0) {
      return fail(MUON_ERR_ALIGNMENT, "%s[%d] = %p is not 16-byte aligned", name, s, p);
    }
    out->p[s] = const_cast<float*>(static_cast<const float*>(p));
  }
  return MUON_OK;
}

muon_status check_ws(const muon_layout* L, const void* ws) {
  if (ws == nullptr) return fail(MUON_ERR_INVALID_ARG, "workspace is NULL");
  if (reinterpret_cast<uintptr_t>(ws) % kWsAlign != 0)
    return fail(MUON_ERR_ALIGNMENT, "workspace %p is not %lld-byte aligned", ws, (long long)kWsAlign);
  (void)L;
  return MUON_OK;
}

muon_status check_full(const void* p, const char* name) {
  if (p == nullptr) return fail(MUON_ERR_INVALID_ARG, "%s is NULL", name);
  if (reinterpret_cast<uintptr_t>(p) % 16 != 0)
    return fail(MUON_ERR_ALIGNMENT, "%s = %p is not 16-byte aligned", name, p);
  return MUON_OK;
}

muon_status check_steps(int32_t ns_steps) {
  if (ns_steps < 0 || ns_steps > 100)
    return fail(MUON_ERR_INVALID_ARG, "ns_steps=%d outside 0..100", ns_steps);
  return MUON_OK;
}

#define MUON_TRY(expr)                    \
  do {                                    \
    const muon_status s_ = (expr);        \
    if (s_ != MUON_OK) return s_;         \
  } while (0)

#define MUON_CUDA(expr, what)                          \
  do {                                                 \
    const cudaError_t e_ = (expr);                     \
    if (e_ != cudaSuccess) return cuda_fail(e_, what); \
  } while (0)

// ---- the three stages (arguments already validated, tables ready) ----
// Hyper-parameters of a call: every group slot holds the same values (ungrouped calls),
// or one slot per optimizer group.
GroupParams uniform_groups(float lr, float wd, float mu, int nesterov) {
  GroupParams gp;
  for (int k = 0; k < kMaxGroups; ++k) {
    gp.lr[k] = lr;
    gp.decay[k] = (float)(1.0 - (double)lr * (double)wd);
    gp.mu[k] = mu;
    gp.nesterov[k] = nesterov ? 1 : 0;
  }
  return gp;
}

muon_status run_momentum(muon_layout* L, const ShardPtrs& g, const ShardPtrs& m, void* ws,
                         const GroupParams& gp, cudaStream_t st) {
  MUON_CUDA(launch_momentum_input(L->plan, L->dt, g, m, ws, gp, st), "momentum_input");
  MUON_CUDA(launch_norm_finalize(L->plan, L->dt, ws, st), "norm_finalize");
  return MUON_OK;
}

muon_status run_ns(muon_layout* L, void* ws, int ns_steps, const ApplyArgs* ap, cudaStream_t st) {
  if (L->plan.ns_dtype != MUON_NS_FP32) {
    MUON_CUDA(launch_ns_tc(L->plan, L->dt, ws, ns_steps, kDefaultBudget, ap, st), "newton_schulz");
    return MUON_OK;
  }
  for (int it = 0; it < ns_steps; ++it)
    for (int ph = 0; ph < 3; ++ph)
      MUON_CUDA(launch_ns_phase_f32(L->plan, L->dt, ws, ph, it & 1, it == 0 ? 1 : 0, st),
                "newton_schulz phase");
  return MUON_OK;
}

// Stages 2 and 3.  On the tensor-core paths with at least one iteration and a fused tail
// (long steps, or MUON_FUSED_TAIL=1) the last Update's epilogue applies
// W <- W*(1 - lr*wd) - lr*scale*O itself, from the fp32 O, and the separate apply pass
// is skipped.
muon_status run_ns_apply(muon_layout* L, const ShardPtrs& w, void* ws, const GroupParams& gp,
                         int ns_steps, cudaStream_t st);

muon_status run_apply(muon_layout* L, const ShardPtrs& w, void* ws, const GroupParams& gp,
                      int ns_steps, cudaStream_t st) {
  MUON_CUDA(launch_apply(L->plan, L->dt, w, ws, ns_steps & 1, ns_steps == 0 ? 1 : 0, gp, st),
            "apply");
  return MUON_OK;
}

muon_status run_ns_apply(muon_layout* L, const ShardPtrs& w, void* ws, const GroupParams& gp,
                         int ns_steps, cudaStream_t st) {
  if (L->plan.ns_dtype != MUON_NS_FP32 && ns_steps >= 1 && L->dt.fused_tail) {
    ApplyArgs ap;
    ap.W = w;
    ap.L = L->plan.L;
    ap.inv_L = 1.0f / (float)L->plan.L;
    ap.gp = gp;
    return run_ns(L, ws, ns_steps, &ap, st);
  }
  muon_status s = run_ns(L, ws, ns_steps, nullptr, st);
  if (s != MUON_OK) return s;
  return run_apply(L, w, ws, gp, ns_steps, st);
}

muon_status check_scalars(float lr, float wd, float mu) {
  if (!std::isfinite(lr) || !std::isfinite(wd) || !std::isfinite(mu))
    return fail(MUON_ERR_INVALID_ARG, "lr, wd and mu must be finite");
  return MUON_OK;
}

}  // namespace

void muon::set_last_error(const std::string& msg) { g_last_error = msg; }

extern "C" {

int32_t muon_abi_version(void) { return MUON_ABI_VERSION; }

const char* muon_last_error(void) { return g_last_error.c_str(); }

muon_status muon_layout_create(const int64_t* shapes, const uint8_t* is_matrix, int32_t n_params,
                               int32_t n_shards, int32_t ns_dtype, muon_layout** out) {
  if (out == nullptr) return fail(MUON_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  muon_layout* L = new (std::nothrow) muon_layout();
  if (L == nullptr) return fail(MUON_ERR_OOM, "out of host memory");
  std::string err;
  try {
    err = build_plan(shapes, is_matrix, n_params, n_shards, ns_dtype, &L->plan);
  } catch (const std::bad_alloc&) {
    delete L;
    return fail(MUON_ERR_OOM, "out of host memory while planning the layout");
  }
  if (!err.empty()) {
    delete L;
    return fail(MUON_ERR_INVALID_ARG, "%s", err.c_str());
  }
  *out = L;
  return ok();
}

muon_status muon_layout_destroy(muon_layout* layout) {
  if (layout == nullptr) return ok();
  free_tables(&layout->dt);
  delete layout;
  return ok();
}

muon_status muon_layout_numel(const muon_layout* layout, int64_t* numel) {
  if (layout == nullptr || numel == nullptr) return fail(MUON_ERR_INVALID_ARG, "NULL argument");
  *numel = layout->plan.N;
  return ok();
}

muon_status muon_layout_shard_len(const muon_layout* layout, int64_t* shard_len) {
  if (layout == nullptr || shard_len == nullptr) return fail(MUON_ERR_INVALID_ARG, "NULL argument");
  *shard_len = layout->plan.L;
  return ok();
}

muon_status muon_layout_workspace_bytes(const muon_layout* layout, size_t* bytes) {
  if (layout == nullptr || bytes == nullptr) return fail(MUON_ERR_INVALID_ARG, "NULL argument");
  *bytes = (size_t)layout->plan.ws_bytes;
  return ok();
}

muon_status muon_layout_full_numel(const muon_layout* layout, int64_t* numel) {
  if (layout == nullptr || numel == nullptr) return fail(MUON_ERR_INVALID_ARG, "NULL argument");
  *numel = layout->plan.full_numel;
  return ok();
}

muon_status muon_full_offsets(const muon_layout* layout, int64_t* offsets) {
  if (layout == nullptr || (offsets == nullptr && layout->plan.n_params > 0))
    return fail(MUON_ERR_INVALID_ARG, "NULL argument");
  for (int32_t i = 0; i < layout->plan.n_params; ++i) offsets[i] = layout->plan.full_off[i];
  return ok();
}

muon_status muon_compute_momentum_inputs(const float* const* flat_grads,
                                         float* const* flat_momentum, const muon_layout* layout,
                                         void* workspace, float mu, int32_t nesterov,
                                         cudaStream_t stream) {
  if (layout == nullptr) return fail(MUON_ERR_INVALID_ARG, "layout is NULL");
  muon_layout* L = const_cast<muon_layout*>(layout);
  ShardPtrs g, m;
  MUON_TRY(check_shards(L, reinterpret_cast<const void* const*>(flat_grads), "flat_grads", &g));
  MUON_TRY(check_shards(L, reinterpret_cast<const void* const*>(flat_momentum), "flat_momentum", &m));
  MUON_TRY(check_ws(L, workspace));
  MUON_TRY(check_scalars(0.f, 0.f, mu));
  std::lock_guard<std::mutex> guard(L->mu);
  MUON_TRY(ensure_device(L));
  MUON_TRY(run_momentum(L, g, m, workspace, uniform_groups(0.f, 0.f, mu, nesterov), stream));
  return ok();
}

muon_status muon_orthogonalize_updates(const muon_layout* layout, void* workspace, int32_t ns_steps,
                                       cudaStream_t stream) {
  if (layout == nullptr) return fail(MUON_ERR_INVALID_ARG, "layout is NULL");
  muon_layout* L = const_cast<muon_layout*>(layout);
  MUON_TRY(check_ws(L, workspace));
  MUON_TRY(check_steps(ns_steps));
  std::lock_guard<std::mutex> guard(L->mu);
  MUON_TRY(ensure_device(L));
  MUON_TRY(ensure_tmaps(L, workspace));
  MUON_TRY(run_ns(L, workspace, ns_steps, nullptr, stream));
  return ok();
}

muon_status muon_orthogonalize_apply(float* const* flat_params, const muon_layout* layout,
                                     void* workspace, float lr, float wd, int32_t ns_steps,
                                     cudaStream_t stream) {
  if (layout == nullptr) return fail(MUON_ERR_INVALID_ARG, "layout is NULL");
  muon_layout* L = const_cast<muon_layout*>(layout);
  ShardPtrs w;
  MUON_TRY(check_shards(L, reinterpret_cast<const void* const*>(flat_params), "flat_params", &w));
  MUON_TRY(check_ws(L, workspace));
  MUON_TRY(check_steps(ns_steps));
  MUON_TRY(check_scalars(lr, wd, 0.f));
  std::lock_guard<std::mutex> guard(L->mu);
  MUON_TRY(ensure_device(L));
  MUON_TRY(ensure_tmaps(L, workspace));
  MUON_TRY(run_ns_apply(L, w, workspace, uniform_groups(lr, wd, 0.f, 0), ns_steps, stream));
  return ok();
}

muon_status muon_apply_local_updates(float* const* flat_params, const muon_layout* layout,
                                     void* workspace, float lr, float wd, int32_t ns_steps,
                                     cudaStream_t stream) {
  if (layout == nullptr) return fail(MUON_ERR_INVALID_ARG, "layout is NULL");
  muon_layout* L = const_cast<muon_layout*>(layout);
  ShardPtrs w;
  MUON_TRY(check_shards(L, reinterpret_cast<const void* const*>(flat_params), "flat_params", &w));
  MUON_TRY(check_ws(L, workspace));
  MUON_TRY(check_steps(ns_steps));
  MUON_TRY(check_scalars(lr, wd, 0.f));
  std::lock_guard<std::mutex> guard(L->mu);
  MUON_TRY(ensure_device(L));
  MUON_TRY(run_apply(L, w, workspace, uniform_groups(lr, wd, 0.f, 0), ns_steps, stream));
  return ok();
}

muon_status muon_step(float* const* flat_params, const float* const* flat_grads,
                      float* const* flat_momentum, const muon_layout* layout, void* workspace,
                      float lr, float wd, float mu, int32_t nesterov, int32_t ns_steps,
                      cudaStream_t stream) {
  if (layout == nullptr) return fail(MUON_ERR_INVALID_ARG, "layout is NULL");
  muon_layout* L = const_cast<muon_layout*>(layout);
  ShardPtrs w, g, m;
  MUON_TRY(check_shards(L, reinterpret_cast<const void* const*>(flat_params), "flat_params", &w));
  MUON_TRY(check_shards(L, reinterpret_cast<const void* const*>(flat_grads), "flat_grads", &g));
  MUON_TRY(check_shards(L, reinterpret_cast<const void* const*>(flat_momentum), "flat_momentum", &m));
  MUON_TRY(check_ws(L, workspace));
  MUON_TRY(check_steps(ns_steps));
  MUON_TRY(check_scalars(lr, wd, mu));
  std::lock_guard<std::mutex> guard(L->mu);
  MUON_TRY(ensure_device(L));
  MUON_TRY(ensure_tmaps(L, workspace));
  const GroupParams gp = uniform_groups(lr, wd, mu, nesterov);
  MUON_TRY(run_momentum(L, g, m, workspace, gp, stream));
  MUON_TRY(run_ns_apply(L, w, workspace, gp, ns_steps, stream));
  return ok();
}

muon_status muon_layout_set_groups(muon_layout* layout, const int32_t* group_of,
                                   int32_t n_groups) {
  if (layout == nullptr) return fail(MUON_ERR_INVALID_ARG, "layout is NULL");
  if (n_groups < 1 || n_groups > kMaxGroups)
    return fail(MUON_ERR_INVALID_ARG, "n_groups=%d outside 1..%d", n_groups, kMaxGroups);
  if (group_of == nullptr && layout->plan.n_params > 0)
    return fail(MUON_ERR_INVALID_ARG, "group_of is NULL");
  for (int32_t i = 0; i < layout->plan.n_params; ++i)
    if (layout->plan.is_matrix[i] && (group_of[i] < 0 || group_of[i] >= n_groups))
      return fail(MUON_ERR_INVALID_ARG, "group_of[%d]=%d outside 0..%d", i, group_of[i],
                  n_groups - 1);
  std::lock_guard<std::mutex> guard(layout->mu);
  for (MatDev& m : layout->plan.mats) m.group = group_of[m.param];
  layout->plan.n_groups = n_groups;
  if (layout->dt.device >= 0 && !layout->plan.mats.empty()) {
    // Tables already on the GPU: refresh the matrix records (synchronous).
    int cur = -1;
    cudaGetDevice(&cur);
    if (cur != layout->dt.device) cudaSetDevice(layout->dt.device);
    const cudaError_t e = cudaMemcpy(layout->dt.mats, layout->plan.mats.data(),
                                     layout->plan.mats.size() * sizeof(MatDev),
                                     cudaMemcpyHostToDevice);
    if (cur >= 0 && cur != layout->dt.device) cudaSetDevice(cur);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(matrix records)");
  }
  return ok();
}

muon_status muon_assign_owners(const muon_layout* layout, int32_t ns_steps, int32_t* owner,
                               double* rank_cost) {
  if (layout == nullptr) return fail(MUON_ERR_INVALID_ARG, "layout is NULL");
  if (owner == nullptr && layout->plan.n_params > 0) return fail(MUON_ERR_INVALID_ARG, "owner is NULL");
  MUON_TRY(check_steps(ns_steps));
  assign_owners(layout->plan, ns_steps, owner, rank_cost);
  return ok();
}

muon_status muon_exchange_plan(const muon_layout* layout, const int32_t* owner, int32_t rank,
                               muon_xfer* sends, int64_t* n_sends, muon_xfer* recvs,
                               int64_t* n_recvs, int64_t* owned_numel, int64_t* owned_offsets) {
  static_assert(sizeof(muon_xfer) == sizeof(XferRun), "muon_xfer and XferRun must agree");
  if (layout == nullptr) return fail(MUON_ERR_INVALID_ARG, "layout is NULL");
  const Plan& plan = layout->plan;
  if (owner == nullptr && plan.n_params > 0) return fail(MUON_ERR_INVALID_ARG, "owner is NULL");
  if (rank < 0 || rank >= plan.n_shards)
    return fail(MUON_ERR_INVALID_ARG, "rank=%d outside 0..%d", rank, plan.n_shards - 1);
  if (n_sends == nullptr || n_recvs == nullptr)
    return fail(MUON_ERR_INVALID_ARG, "n_sends and n_recvs must not be NULL");
  std::vector<XferRun> runs;
  std::vector<int64_t> offs, owned;
  const std::string err = exchange_runs(plan, owner, &runs, &offs, &owned);
  if (!err.empty()) return fail(MUON_ERR_INVALID_ARG, "%s", err.c_str());
  std::vector<XferRun> snd, rcv;
  for (const XferRun& r : runs) {
    if (r.src_rank == rank) snd.push_back(r);
    if (r.dst_rank == rank) rcv.push_back(r);
  }
  // runs come in (parameter, offset) order; a stable sort by peer keeps it within a peer
  std::stable_sort(snd.begin(), snd.end(),
                   [](const XferRun& a, const XferRun& b) { return a.dst_rank < b.dst_rank; });
  std::stable_sort(rcv.begin(), rcv.end(),
                   [](const XferRun& a, const XferRun& b) { return a.src_rank < b.src_rank; });
  if (sends != nullptr && *n_sends < (int64_t)snd.size())
    return fail(MUON_ERR_INVALID_ARG, "sends holds %lld runs, %zu needed", (long long)*n_sends,
                snd.size());
  if (recvs != nullptr && *n_recvs < (int64_t)rcv.size())
    return fail(MUON_ERR_INVALID_ARG, "recvs holds %lld runs, %zu needed", (long long)*n_recvs,
                rcv.size());
  if (sends != nullptr) std::memcpy(sends, snd.data(), snd.size() * sizeof(XferRun));
  if (recvs != nullptr) std::memcpy(recvs, rcv.data(), rcv.size() * sizeof(XferRun));
  *n_sends = (int64_t)snd.size();
  *n_recvs = (int64_t)rcv.size();
  if (owned_numel != nullptr) *owned_numel = owned[rank];
  if (owned_offsets != nullptr)
    for (int32_t i = 0; i < plan.n_params; ++i) owned_offsets[i] = offs[i];
  return ok();
}

muon_status muon_step_grouped(float* const* flat_params, const float* const* flat_grads,
                              float* const* flat_momentum, const muon_layout* layout,
                              void* workspace, const muon_group_hparams* groups, int32_t ns_steps,
                              cudaStream_t stream) {
  if (layout == nullptr) return fail(MUON_ERR_INVALID_ARG, "layout is NULL");
  muon_layout* L = const_cast<muon_layout*>(layout);
  if (groups == nullptr) return fail(MUON_ERR_INVALID_ARG, "groups is NULL");
  ShardPtrs w, g, m;
  MUON_TRY(check_shards(L, reinterpret_cast<const void* const*>(flat_params), "flat_params", &w));
  MUON_TRY(check_shards(L, reinterpret_cast<const void* const*>(flat_grads), "flat_grads", &g));
  MUON_TRY(check_shards(L, reinterpret_cast<const void* const*>(flat_momentum), "flat_momentum", &m));
  MUON_TRY(check_ws(L, workspace));
  MUON_TRY(check_steps(ns_steps));
  GroupParams gp = uniform_groups(0.f, 0.f, 0.f, 0);
  for (int k = 0; k < L->plan.n_groups; ++k) {
    MUON_TRY(check_scalars(groups[k].lr, groups[k].wd, groups[k].mu));
    gp.lr[k] = groups[k].lr;
    gp.decay[k] = (float)(1.0 - (double)groups[k].lr * (double)groups[k].wd);
    gp.mu[k] = groups[k].mu;
    gp.nesterov[k] = groups[k].nesterov != 0 ? 1 : 0;
  }
  std::lock_guard<std::mutex> guard(L->mu);
  MUON_TRY(ensure_device(L));
  MUON_TRY(ensure_tmaps(L, workspace));
  MUON_TRY(run_momentum(L, g, m, workspace, gp, stream));
  MUON_TRY(run_ns_apply(L, w, workspace, gp, ns_steps, stream));
  return ok();
}

muon_status muon_gather_full(const muon_layout* layout, const float* const* shards, float* full,
                             cudaStream_t stream) {
  if (layout == nullptr) return fail(MUON_ERR_INVALID_ARG, "layout is NULL");
  muon_layout* L = const_cast<muon_layout*>(layout);
  ShardPtrs s;
  MUON_TRY(check_shards(L, reinterpret_cast<const void* const*>(shards), "shards", &s));
  if (L->plan.full_numel > 0) MUON_TRY(check_full(full, "full"));
  std::lock_guard<std::mutex> guard(L->mu);
  MUON_TRY(ensure_device(L));
  MUON_CUDA(launch_gather(L->plan, L->dt, s, full, stream), "gather");
  return ok();
}

muon_status muon_scatter_updates(const muon_layout* layout, const float* full, float* const* shards,
                                 cudaStream_t stream) {
  if (layout == nullptr) return fail(MUON_ERR_INVALID_ARG, "layout is NULL");
  muon_layout* L = const_cast<muon_layout*>(layout);
  ShardPtrs s;
  MUON_TRY(check_shards(L, reinterpret_cast<const void* const*>(shards), "shards", &s));
  if (L->plan.full_numel > 0) MUON_TRY(check_full(full, "full"));
  std::lock_guard<std::mutex> guard(L->mu);
  MUON_TRY(ensure_device(L));
  MUON_CUDA(launch_scatter(L->plan, L->dt, full, s, stream), "scatter");
  return ok();
}

muon_status muon_orthogonalize_full(const muon_layout* layout, void* workspace, const float* full_in,
                                    float* full_out, int32_t ns_steps, cudaStream_t stream) {
  if (layout == nullptr) return fail(MUON_ERR_INVALID_ARG, "layout is NULL");
  muon_layout* L = const_cast<muon_layout*>(layout);
  MUON_TRY(check_ws(L, workspace));
  MUON_TRY(check_steps(ns_steps));
  if (L->plan.full_numel > 0) {
    MUON_TRY(check_full(full_in, "full_in"));
    MUON_TRY(check_full(full_out, "full_out"));
  }
  std::lock_guard<std::mutex> guard(L->mu);
  MUON_TRY(ensure_device(L));
  MUON_TRY(ensure_tmaps(L, workspace));
  MUON_CUDA(launch_full_input(L->plan, L->dt, full_in, workspace, stream), "full_input");
  MUON_CUDA(launch_norm_finalize(L->plan, L->dt, workspace, stream), "norm_finalize");
  MUON_TRY(run_ns(L, workspace, ns_steps, nullptr, stream));
  MUON_CUDA(launch_export(L->plan, L->dt, workspace, ns_steps & 1, ns_steps == 0 ? 1 : 0, full_out,
                          stream),
            "export");
  return ok();
}

muon_status muon_export_input(const muon_layout* layout, const void* workspace, float* full_out,
                              cudaStream_t stream) {
  if (layout == nullptr) return fail(MUON_ERR_INVALID_ARG, "layout is NULL");
  muon_layout* L = const_cast<muon_layout*>(layout);
  MUON_TRY(check_ws(L, workspace));
  if (L->plan.full_numel > 0) MUON_TRY(check_full(full_out, "full_out"));
  std::lock_guard<std::mutex> guard(L->mu);
  MUON_TRY(ensure_device(L));
  MUON_CUDA(launch_export(L->plan, L->dt, workspace, 0, 0, full_out, stream), "export");
  return ok();
}

muon_status muon_export_update(const muon_layout* layout, const void* workspace, int32_t ns_steps,
                               float* full_out, cudaStream_t stream) {
  if (layout == nullptr) return fail(MUON_ERR_INVALID_ARG, "layout is NULL");
  muon_layout* L = const_cast<muon_layout*>(layout);
  MUON_TRY(check_ws(L, workspace));
  MUON_TRY(check_steps(ns_steps));
  if (L->plan.full_numel > 0) MUON_TRY(check_full(full_out, "full_out"));
  std::lock_guard<std::mutex> guard(L->mu);
  MUON_TRY(ensure_device(L));
  MUON_CUDA(launch_export(L->plan, L->dt, workspace, ns_steps & 1, ns_steps == 0 ? 1 : 0,
                          full_out, stream),
            "export");
  return ok();
}

muon_status muon_check(cudaStream_t stream) {
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  int dev = -1;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  int* word = nullptr;
  MUON_TRY(err_word(dev, &word));
  int h = 0;
  e = cudaMemcpy(&h, word, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(error word)");
  // The allocation-free entry point keeps its own error word in its scratch array.
  int h2 = 0;
  int* word2 = noalloc_error_word(dev);
  if (word2 != nullptr) {
    e = cudaMemcpy(&h2, word2, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(error word)");
    if (h2 != 0) cudaMemset(word2, 0, sizeof(int));
  }
  if (h == 0) h = h2;
  if (h != 0) {
    cudaMemset(word, 0, sizeof(int));
    if (h == MUON_ERR_TIMEOUT)
      return fail(MUON_ERR_TIMEOUT, "a device-side wait ran out of its budget and the kernel exited");
    if (h == MUON_ERR_DEVICE_CHECK)
      return fail(MUON_ERR_DEVICE_CHECK, "a device-side range check of a table entry failed "
                  "(debug build); the work it drove was skipped");
    return fail(MUON_ERR_CUDA, "device error word %d", h);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "pending CUDA error");
  return ok();
}

muon_status muon_layout_ns_kernel(const muon_layout* layout, int32_t* tile_shape, int32_t* units,
                                  int32_t* persistent) {
  if (layout == nullptr || tile_shape == nullptr || units == nullptr || persistent == nullptr)
    return fail(MUON_ERR_INVALID_ARG, "null argument");
  muon_layout* L = const_cast<muon_layout*>(layout);
  std::lock_guard<std::mutex> guard(L->mu);
  MUON_TRY(ensure_device(L));
  const bool tc = L->plan.ns_dtype != MUON_NS_FP32 && !L->plan.mats.empty();
  *tile_shape = tc ? L->dt.tc_shape : 0;
  *units = tc ? L->dt.tc_units : 0;
  *persistent = tc && L->dt.tc_persistent ? 1 : 0;
  return ok();
}

muon_status muon_layout_fused_apply(const muon_layout* layout, int32_t* fused) {
  if (layout == nullptr || fused == nullptr) return fail(MUON_ERR_INVALID_ARG, "null argument");
  muon_layout* L = const_cast<muon_layout*>(layout);
  std::lock_guard<std::mutex> guard(L->mu);
  MUON_TRY(ensure_device(L));
  const bool tc = L->plan.ns_dtype != MUON_NS_FP32 && !L->plan.mats.empty();
  *fused = tc && L->dt.fused_tail ? 1 : 0;
  return ok();
}

int32_t muon_debug_build(void) { return kDebugChecks ? 1 : 0; }

muon_status muon_selftest_device_check(cudaStream_t stream) {
  if (!kDebugChecks)
    return fail(MUON_ERR_UNSUPPORTED, "this library was built without -DMUON_DEBUG");
  int dev = -1;
  MUON_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // One 2 x 4 matrix and one chunk of 16 elements: longer than the matrix, so the check
  // must refuse it.  Shard and full buffers hold 64 floats, so even an unchecked copy of
  // the chunk would stay inside them.
  Plan plan;
  plan.n_params = 1;
  plan.n_shards = 1;
  plan.ns_dtype = MUON_NS_FP32;
  plan.N = 8;
  plan.L = 16;
  plan.full_numel = 8;
  plan.ws_bytes = 1 << 20;
  MatDev m{};
  m.rows = 2; m.cols = 4; m.m = 2; m.n = 4; m.tall = 0; m.ldx = 8; m.lda = 8;
  m.scale = 1.f; m.chunk_begin = 0; m.chunk_end = 1;
  ChunkDev c{};
  c.mat = 0; c.shard = 0; c.shard_off = 0; c.local = 0; c.len = 16; c.vec = 1;
  plan.mats.push_back(m);
  plan.chunks.push_back(c);
  uint8_t* buf = nullptr;
  const size_t bytes = 256 + 256 + 2 * 64 * sizeof(float);
  MUON_CUDA(cudaMalloc(&buf, bytes), "cudaMalloc(selftest tables)");
  cudaMemsetAsync(buf, 0, bytes, stream);
  cudaMemcpyAsync(buf, &c, sizeof(c), cudaMemcpyHostToDevice, stream);
  cudaMemcpyAsync(buf + 256, &m, sizeof(m), cudaMemcpyHostToDevice, stream);
  DevTables dt;
  dt.device = dev;
  dt.n_sms = sms;
  muon_status st = err_word(dev, &dt.err);
  if (st != MUON_OK) { cudaFree(buf); return st; }
  dt.chunks = reinterpret_cast<ChunkDev*>(buf);
  dt.mats = reinterpret_cast<MatDev*>(buf + 256);
  ShardPtrs sp;
  std::memset(&sp, 0, sizeof(sp));
  sp.p[0] = reinterpret_cast<float*>(buf + 512);
  float* full = reinterpret_cast<float*>(buf + 512 + 64 * sizeof(float));
  cudaError_t e = launch_gather(plan, dt, sp, full, stream);
  const cudaError_t e2 = cudaStreamSynchronize(stream);
  cudaFree(buf);
  if (e != cudaSuccess) return cuda_fail(e, "selftest gather");
  if (e2 != cudaSuccess) return cuda_fail(e2, "cudaStreamSynchronize");
  return ok();
}

muon_status muon_selftest_wait_timeout(int64_t budget_cycles, cudaStream_t stream) {
  if (budget_cycles < 1 || budget_cycles > ((int64_t)1 << 40))
    return fail(MUON_ERR_INVALID_ARG, "budget_cycles outside 1..2^40");
  int dev = -1;
  MUON_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  int* word = nullptr;
  MUON_TRY(err_word(dev, &word));
  MUON_CUDA(launch_selftest_timeout(word, (long long)budget_cycles, stream), "selftest");
  return ok();
}

}  // extern "C"
