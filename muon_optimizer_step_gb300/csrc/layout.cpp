// Host planner: where every parameter lives in the flat buffer and its shards, the
// per-matrix full layout, the chunk table of the streaming kernels, the workspace map
// and the per-phase tile work lists of the Newton-Schulz GEMMs.
//
// Flat packing follows "Add initial Muon+M-FSDPv2 implementation" ("What does this PR
// do?": every parameter in flat shards): parameters back to back in the caller's order, no padding,
// shard s of n_shards holding flat [s*L, (s+1)*L) with L = ceil(N / n_shards).  Matrix
// parameters may straddle any number of shard edges; the gather and scatter of the
// owner ("Opt step" steps 3 and 5) are then the index map built here.
#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdio>
#include <numeric>
#include <queue>

#include "muon_internal.h"

namespace muon {

namespace {

int64_t round_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

std::string fmt(const char* f, long long a, long long b = 0, long long c = 0) {
  char buf[256];
  std::snprintf(buf, sizeof(buf), f, a, b, c);
  return buf;
}

}  // namespace

std::string build_plan(const int64_t* shapes, const uint8_t* is_matrix, int32_t n_params,
                       int32_t n_shards, int32_t ns_dtype, Plan* plan) {
  if (n_params < 0) return "n_params must be >= 0";
  if (n_params > 0 && shapes == nullptr) return "shapes is NULL";
  if (n_shards < 1 || n_shards > 128) return fmt("n_shards=%lld outside 1..128", n_shards);
  if (ns_dtype < 0 || ns_dtype > 2)
    return fmt("ns_dtype=%lld is not 0 (bf16), 1 (fp32) or 2 (split fp32)", ns_dtype);
  Plan p;
  p.n_params = n_params;
  p.n_shards = n_shards;
  p.ns_dtype = ns_dtype;
  p.rows.resize(n_params);
  p.cols.resize(n_params);
  p.is_matrix.resize(n_params);
  p.flat_off.resize(n_params);
  p.full_off.assign(n_params, -1);
  const int64_t kMaxFlat = (int64_t)1 << 46;
  int64_t pos = 0, full = 0;
  for (int32_t i = 0; i < n_params; ++i) {
    const int64_t r = shapes[2 * i], c = shapes[2 * i + 1];
    const bool mat = is_matrix ? is_matrix[i] != 0 : true;
    p.rows[i] = r;
    p.cols[i] = c;
    p.is_matrix[i] = mat ? 1 : 0;
    if (mat) {
      if (r < 1 || c < 1) return fmt("matrix parameter %lld has shape %lld x %lld", i, r, c);
      if (r > INT32_MAX / c) return fmt("matrix parameter %lld (%lld x %lld) exceeds 2^31-1 elements", i, r, c);
    } else {
      if (r < 0 || c < 0) return fmt("parameter %lld has negative shape %lld x %lld", i, r, c);
      if (c != 0 && r > kMaxFlat / c) return fmt("parameter %lld (%lld x %lld) is too large", i, r, c);
    }
    p.flat_off[i] = pos;
    pos += r * c;
    if (pos > kMaxFlat) return "flat buffer exceeds 2^46 elements";
    if (mat) {
      full = round_up(full, 4);
      p.full_off[i] = full;
      full += r * c;
    }
  }
  p.N = pos;
  p.L = (pos + n_shards - 1) / n_shards;
  p.full_numel = full;

  // Matrices, their workspace buffers and chunk tables.
  const int64_t esz = ns_dtype == 1 ? 4 : 2;
  const int64_t parts = ns_dtype == 2 ? 3 : 1;  // split fp32: h, m and l bf16 arrays
  int64_t n_mats = 0;
  for (int32_t i = 0; i < n_params; ++i) n_mats += p.is_matrix[i];
  int64_t n_chunks = 0;
  for (int32_t i = 0; i < n_params; ++i) {
    if (!p.is_matrix[i]) continue;
    MatDev m{};
    m.rows = (int32_t)p.rows[i];
    m.cols = (int32_t)p.cols[i];
    m.m = std::min(m.rows, m.cols);
    m.n = std::max(m.rows, m.cols);
    m.tall = m.rows > m.cols ? 1 : 0;
    m.ldx = (int32_t)round_up(m.cols, 8);
    m.lda = (int32_t)round_up(m.m, 8);
    m.param = i;
    m.full_off = p.full_off[i];
    m.flat_off = p.flat_off[i];
    m.scale = (float)std::sqrt(std::max(1.0, (double)m.rows / (double)m.cols));
    m.group = 0;
    m.chunk_begin = (int64_t)p.chunks.size();
    const int64_t numel = (int64_t)m.rows * m.cols;
    const bool dense_x = (m.ldx == m.cols);
    // Chunks are cut at fixed multiples of kChunkElems of the matrix's own row-major
    // index, never at shard edges: the per-chunk sums of squares (and so ||X||) are then
    // the same bits for every sharding of the same buffer.  A chunk that crosses a shard
    // edge takes the kernels' per-element path.
    int64_t local = 0;
    while (local < numel) {
      const int64_t g = p.flat_off[i] + local;
      const int64_t s = g / p.L;
      const int64_t so = g - s * p.L;
      const int64_t len = std::min<int64_t>(kChunkElems, numel - local);
      ChunkDev ch{};
      ch.mat = (int32_t)p.mats.size();
      ch.shard = (int32_t)s;
      ch.shard_off = so;
      ch.local = local;
      ch.len = (int32_t)len;
      const bool one_shard = so + len <= p.L;
      ch.vec = (one_shard && so % 4 == 0 && local % 4 == 0 && m.full_off % 4 == 0 && dense_x)
                   ? 1 : 0;
      p.chunks.push_back(ch);
      local += len;
    }
    m.chunk_end = (int64_t)p.chunks.size();
    n_chunks = (int64_t)p.chunks.size();
    p.mats.push_back(m);
  }
  (void)n_mats;
  int64_t ws = 0;
  p.ws_partials = ws;
  ws += n_chunks * 4;
  ws = round_up(ws, 16);
  p.ws_inv_norm = ws;
  ws += (int64_t)p.mats.size() * 4;
  ws = round_up(ws, 16);
  p.ws_counters = ws;
  ws += (int64_t)p.mats.size() * 3 * 4;
  ws = round_up(ws, kWsAlign);
  for (MatDev& m : p.mats) {
    const int64_t xb = round_up((int64_t)m.rows * m.ldx * esz, kWsAlign) * parts;
    const int64_t ab = round_up((int64_t)m.m * m.lda * esz, kWsAlign) * parts;
    m.x0 = ws; ws += xb;
    m.x1 = ws; ws += xb;
    m.a = ws; ws += ab;
    m.b = ws; ws += ab;
  }
  p.ws_bytes = std::max<int64_t>(ws, kWsAlign);
  *plan = std::move(p);
  return "";
}

namespace {

struct Item {
  TileDev t;
  int64_t cost;  // k-blocks plus an epilogue allowance
};

// The output tiles of one phase over every matrix, in matrix order.
std::vector<Item> phase_items(const Plan& plan, int phase, int bm, int bn, int bk) {
  std::vector<Item> items;
  for (size_t mi = 0; mi < plan.mats.size(); ++mi) {
    const MatDev& m = plan.mats[mi];
    int M, N, K;
    bool sym;
    if (phase == kPhaseGram) { M = N = m.m; K = m.n; sym = true; }
    else if (phase == kPhasePoly) { M = N = m.m; K = m.m; sym = true; }
    else { M = m.rows; N = m.cols; K = m.m; sym = false; }
    const int kb = (K + bk - 1) / bk;
    // Tile order = the order in which a wave of CTAs picks tiles up (equal-cost tiles are
    // dealt round-robin).  The Update of a wide matrix (B X: X panels along j, B m x m)
    // walks j in the outer loop so that each X column panel is read from HBM once while
    // B stays in L2; every other phase walks rows (i) outermost, which for a tall Update
    // (X B) streams each X row panel once against the L2-resident B.
    const bool j_outer = phase == kPhaseUpdate && !m.tall;
    const int outer = j_outer ? N : M, inner = j_outer ? M : N;
    const int ostep = j_outer ? bn : bm, istep = j_outer ? bm : bn;
    for (int o0 = 0; o0 < outer; o0 += ostep) {
      for (int n0 = 0; n0 < inner; n0 += istep) {
        const int i0 = j_outer ? n0 : o0, j0 = j_outer ? o0 : n0;
        // Symmetric outputs: only tiles that reach the upper triangle (col >= row).
        if (sym && j0 + bn - 1 < i0) continue;
        Item it;
        it.t.mat = (int32_t)mi;
        it.t.i0 = i0;
        it.t.j0 = j0;
        it.t.kblocks = kb;
        it.cost = (int64_t)kb + (sym ? 3 : 2);
        items.push_back(it);
      }
    }
  }
  return items;
}

// Heap of units by the cost-time at which they free up (lowest index on ties).
using Slot = std::pair<int64_t, int>;
using SlotHeap = std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>>;

TileList pack_lists(std::vector<std::vector<TileDev>>& per, int grid) {
  TileList tl;
  tl.grid = grid;
  tl.cta_begin.resize(grid + 1);
  tl.cta_begin[0] = 0;
  for (int c = 0; c < grid; ++c) {
    tl.cta_begin[c + 1] = tl.cta_begin[c] + (int32_t)per[c].size();
    tl.tiles.insert(tl.tiles.end(), per[c].begin(), per[c].end());
  }
  return tl;
}

}  // namespace

TileList plan_tiles(const Plan& plan, int phase, int bm, int bn, int bk, int n_sms,
                    bool by_cost) {
  std::vector<Item> items = phase_items(plan, phase, bm, bn, bk);
  if (by_cost)
    std::stable_sort(items.begin(), items.end(),
                     [](const Item& a, const Item& b) { return a.cost > b.cost; });
  if (items.empty() || n_sms <= 0) {
    TileList tl;
    tl.grid = 0;
    tl.cta_begin.assign(1, 0);
    return tl;
  }
  const int grid = (int)std::min<int64_t>((int64_t)items.size(), n_sms);
  // LPT: each tile, most expensive first, goes to the least-loaded CTA (lowest index on ties).
  SlotHeap heap;
  for (int c = 0; c < grid; ++c) heap.push({0, c});
  std::vector<std::vector<TileDev>> per(grid);
  for (const Item& it : items) {
    Slot s = heap.top();
    heap.pop();
    per[s.second].push_back(it.t);
    heap.push({s.first + it.cost, s.second});
  }
  return pack_lists(per, grid);
}

std::vector<TileList> plan_persistent(const Plan& plan, int bm, int bn, int bk, int units,
                                      int iters) {
  std::vector<TileList> out;
  if (units <= 0 || iters <= 0) return out;
  std::vector<Item> items[3];
  for (int ph = 0; ph < 3; ++ph) items[ph] = phase_items(plan, ph, bm, bn, bk);
  const size_t nm = plan.mats.size();
  std::vector<int64_t> ready(nm, 0), done(nm, 0);
  SlotHeap heap;
  for (int u = 0; u < units; ++u) heap.push({0, u});
  for (int q = 0; q < 3 * iters; ++q) {
    const std::vector<Item>& it = items[q % 3];
    std::vector<size_t> order(it.size());
    std::iota(order.begin(), order.end(), size_t{0});
    std::stable_sort(order.begin(), order.end(), [&](size_t a, size_t b) {
      const int64_t ra = ready[it[a].t.mat], rb = ready[it[b].t.mat];
      return ra != rb ? ra < rb : it[a].cost > it[b].cost;
    });
    std::vector<std::vector<TileDev>> per(units);
    std::vector<std::vector<int64_t>> end(units);
    for (size_t k : order) {
      const Item& x = it[k];
      const Slot s = heap.top();
      heap.pop();
      const int64_t start = std::max(s.first, ready[x.t.mat]);
      per[s.second].push_back(x.t);
      end[s.second].push_back(start + x.cost);
      heap.push({start + x.cost, s.second});
    }
    // A tile is published when the next tile of its list ends (the last one when it ends).
    std::fill(done.begin(), done.end(), 0);
    for (int u = 0; u < units; ++u) {
      const size_t n = per[u].size();
      for (size_t i = 0; i < n; ++i) {
        const int64_t pub = end[u][i + 1 < n ? i + 1 : i] + kPublishLag;
        done[per[u][i].mat] = std::max(done[per[u][i].mat], pub);
      }
    }
    ready.swap(done);
    out.push_back(pack_lists(per, units));
  }
  return out;
}

void assign_owners(const Plan& plan, int ns_steps, int32_t* owner, double* rank_cost) {
  const int S = plan.n_shards;
  std::vector<double> load(S, 0.0);
  struct Job { double cost; int32_t param; int64_t first, last; };
  std::vector<Job> jobs;
  for (int32_t i = 0; i < plan.n_params; ++i) {
    owner[i] = -1;
    if (!plan.is_matrix[i]) continue;
    const double r = (double)plan.rows[i], c = (double)plan.cols[i];
    const double m = std::min(r, c), n = std::max(r, c);
    Job j;
    j.cost = (double)ns_steps * (3.0 * m * m * n + m * m * m);
    j.param = i;
    const int64_t numel = plan.rows[i] * plan.cols[i];
    j.first = plan.flat_off[i] / plan.L;
    j.last = (plan.flat_off[i] + numel - 1) / plan.L;
    jobs.push_back(j);
  }
  // Most expensive first; equal costs keep the parameters' order.
  std::stable_sort(jobs.begin(), jobs.end(),
                   [](const Job& a, const Job& b) { return a.cost > b.cost; });
  for (const Job& j : jobs) {
    int64_t best = j.first;
    for (int64_t s = j.first + 1; s <= j.last; ++s)
      if (load[s] < load[best]) best = s;
    owner[j.param] = (int32_t)best;
    load[best] += j.cost;
  }
  if (rank_cost != nullptr)
    for (int s = 0; s < S; ++s) rank_cost[s] = load[s];
}

std::string exchange_runs(const Plan& plan, const int32_t* owner, std::vector<XferRun>* runs,
                          std::vector<int64_t>* owner_offsets, std::vector<int64_t>* owned_numel) {
  const int S = plan.n_shards;
  runs->clear();
  owner_offsets->assign(plan.n_params, -1);
  owned_numel->assign(S, 0);
  for (int32_t i = 0; i < plan.n_params; ++i) {
    if (!plan.is_matrix[i]) continue;
    const int32_t o = owner[i];
    if (o < 0 || o >= S)
      return fmt("owner[%lld]=%lld outside 0..%lld", i, o, S - 1);
    // The owner's packed buffer: its parameters in order, each at a multiple of 4.
    int64_t& end = (*owned_numel)[o];
    end = round_up(end, 4);
    (*owner_offsets)[i] = end;
    const int64_t numel = plan.rows[i] * plan.cols[i];
    // Cut [flat_off, flat_off + numel) at shard edges.
    int64_t g = plan.flat_off[i];
    const int64_t g_end = g + numel;
    while (g < g_end) {
      const int64_t s = g / plan.L;
      const int64_t edge = std::min(g_end, (s + 1) * plan.L);
      XferRun r{};
      r.param = i;
      r.src_rank = (int32_t)s;
      r.dst_rank = o;
      r.shard_off = g - s * plan.L;
      r.owner_off = end + (g - plan.flat_off[i]);
      r.len = edge - g;
      runs->push_back(r);
      g = edge;
    }
    end += numel;
  }
  return "";
}

}  // namespace muon
