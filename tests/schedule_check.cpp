// Host check of the Newton-Schulz tile planner (muon_optimizer_step_gb300/csrc/layout.cpp),
// compiled with g++ and run by test_schedule.py.  For several matrix sets, tile shapes and
// unit counts it checks that:
//  - every list (per phase, or per iteration and phase for a persistent launch) holds each
//    tile of its phase exactly once, with well-formed per-unit offsets;
//  - the persistent lists do not depend on how many iterations were planned;
//  - a run that follows the kernel's waiting rules (a tile waits until every tile of its
//    matrix's previous phase is published; a tile is published when the next tile of its
//    list has run, or at once when it is the last) finishes every tile, whatever order the
//    units take turns in and whatever each tile costs;
//  - on GPT-2-small shapes, the timed run of those rules with the planner's cost model
//    ends no later with the persistent lists than with per-phase lists in matrix order.
#include <algorithm>
#include <cstdio>
#include <random>
#include <string>
#include <tuple>
#include <vector>

#include "muon_internal.h"

using namespace muon;

namespace {

int g_failures = 0;

#define CHECK(cond, ...)                                            \
  do {                                                              \
    if (!(cond)) {                                                  \
      ++g_failures;                                                 \
      std::printf("FAIL line %d: ", __LINE__);                      \
      std::printf(__VA_ARGS__);                                     \
      std::printf("\n");                                            \
    }                                                               \
  } while (0)

using Shapes = std::vector<std::pair<int64_t, int64_t>>;
using Key = std::tuple<int, int, int, int>;

Plan make_plan(const Shapes& shapes) {
  std::vector<int64_t> sh;
  std::vector<uint8_t> im;
  for (const auto& s : shapes) {
    sh.push_back(s.first);
    sh.push_back(s.second);
    im.push_back(1);
  }
  Plan p;
  const std::string e = build_plan(sh.data(), im.data(), (int32_t)shapes.size(), 1, 0, &p);
  CHECK(e.empty(), "build_plan: %s", e.c_str());
  return p;
}

std::vector<Key> sorted_keys(const std::vector<TileDev>& v) {
  std::vector<Key> k;
  for (const TileDev& t : v) k.emplace_back(t.mat, t.i0, t.j0, t.kblocks);
  std::sort(k.begin(), k.end());
  return k;
}

bool same_lists(const TileList& a, const TileList& b) {
  if (a.cta_begin != b.cta_begin || a.tiles.size() != b.tiles.size()) return false;
  for (size_t i = 0; i < a.tiles.size(); ++i)
    if (a.tiles[i].mat != b.tiles[i].mat || a.tiles[i].i0 != b.tiles[i].i0 ||
        a.tiles[i].j0 != b.tiles[i].j0 || a.tiles[i].kblocks != b.tiles[i].kblocks)
      return false;
  return true;
}

// The lists of q = 0 .. 3*iters-1 as one launch walks them: list q, or the last
// iteration's list of the same phase past the planned ones.
const TileList& list_of(const std::vector<TileList>& lists, int q) {
  const int n = (int)lists.size();
  return lists[q < n ? q : n - 3 + q % 3];
}

void check_well_formed(const TileList& tl, int units, const std::vector<Key>& want,
                       const char* what) {
  CHECK((int)tl.cta_begin.size() == units + 1, "%s: %zu offsets for %d units", what,
        tl.cta_begin.size(), units);
  if ((int)tl.cta_begin.size() != units + 1) return;
  CHECK(tl.cta_begin[0] == 0 && tl.cta_begin[units] == (int32_t)tl.tiles.size(),
        "%s: offsets do not span the list", what);
  for (int u = 0; u < units; ++u)
    CHECK(tl.cta_begin[u] <= tl.cta_begin[u + 1], "%s: offsets decrease at unit %d", what, u);
  CHECK(sorted_keys(tl.tiles) == want, "%s: not every tile of the phase exactly once", what);
}

// Runs the kernel's waiting rules over `iters` iterations.  Returns the number of tiles
// run (all of them unless the rules deadlock) and, with costs, the time the last one is
// published.  order_seed < 0: the runnable unit with the earliest start goes next (a timed
// run); otherwise a random runnable unit (an untimed run with random tile costs).
struct RunResult {
  int64_t tiles_run = 0, tiles_total = 0;
  double makespan = 0.0;
};

RunResult run_rules(const Plan& plan, const std::vector<TileList>& lists, int units, int iters,
                    int order_seed) {
  const int nq = 3 * iters;
  const size_t nm = plan.mats.size();
  std::vector<std::vector<int>> total(nq, std::vector<int>(nm, 0));
  std::vector<std::vector<int>> published(nq, std::vector<int>(nm, 0));
  std::vector<std::vector<double>> pub_time(nq, std::vector<double>(nm, 0.0));
  RunResult r;
  for (int q = 0; q < nq; ++q)
    for (const TileDev& t : list_of(lists, q).tiles) {
      ++total[q][t.mat];
      ++r.tiles_total;
    }
  std::vector<int> uq(units, 0), ui(units, 0);
  std::vector<double> free_at(units, 0.0), prev_end(units, 0.0);
  std::vector<int> prev_mat(units, -1);
  std::mt19937 rng(order_seed < 0 ? 1u : (unsigned)order_seed);
  std::uniform_real_distribution<double> jitter(0.25, 4.0);
  auto publish = [&](int q, int mat, double t) {
    ++published[q][mat];
    pub_time[q][mat] = std::max(pub_time[q][mat], t);
  };
  while (true) {
    int best = -1;
    double best_start = 0.0;
    std::vector<int> runnable;
    for (int u = 0; u < units; ++u) {
      // skip finished lists (publishing their last tile has already happened)
      while (uq[u] < nq) {
        const TileList& tl = list_of(lists, uq[u]);
        if (tl.cta_begin[u] + ui[u] < tl.cta_begin[u + 1]) break;
        ++uq[u];
        ui[u] = 0;
      }
      if (uq[u] >= nq) continue;
      const int q = uq[u];
      const TileList& tl = list_of(lists, q);
      const TileDev& t = tl.tiles[tl.cta_begin[u] + ui[u]];
      double dep = 0.0;
      if (q > 0) {
        if (published[q - 1][t.mat] < total[q - 1][t.mat]) continue;
        dep = pub_time[q - 1][t.mat];
      }
      const double start = std::max(free_at[u], dep);
      runnable.push_back(u);
      if (best < 0 || start < best_start) {
        best = u;
        best_start = start;
      }
    }
    if (runnable.empty()) break;
    int u = best;
    if (order_seed >= 0) u = runnable[rng() % runnable.size()];
    const int q = uq[u];
    const TileList& tl = list_of(lists, q);
    const TileDev& t = tl.tiles[tl.cta_begin[u] + ui[u]];
    const double cost = (double)t.kblocks + (q % 3 == kPhaseUpdate ? 2.0 : 3.0);
    const double start = order_seed >= 0 ? 0.0 : best_start;
    const double end = start + (order_seed >= 0 ? cost * jitter(rng) : cost);
    if (ui[u] > 0) publish(q, prev_mat[u], end + (double)kPublishLag);
    const bool last = tl.cta_begin[u] + ui[u] + 1 >= tl.cta_begin[u + 1];
    if (last) publish(q, t.mat, end + (double)kPublishLag);
    prev_mat[u] = t.mat;
    free_at[u] = end;
    ++ui[u];
    ++r.tiles_run;
    r.makespan = std::max(r.makespan, end + (double)kPublishLag);
  }
  return r;
}

void check_set(const char* name, const Shapes& shapes, int bm, int bn, int units, bool timed) {
  const Plan plan = make_plan(shapes);
  if (plan.mats.empty()) return;
  std::vector<Key> want[3];
  std::vector<TileList> per_phase;
  for (int p = 0; p < 3; ++p) {
    per_phase.push_back(plan_tiles(plan, p, bm, bn, kTcBK, units));
    want[p] = sorted_keys(per_phase.back().tiles);
    CHECK(!want[p].empty(), "%s: phase %d has no tiles", name, p);
  }
  const int iters = 6;
  const std::vector<TileList> pers = plan_persistent(plan, bm, bn, kTcBK, units, iters);
  CHECK((int)pers.size() == 3 * iters, "%s: %zu persistent lists", name, pers.size());
  if ((int)pers.size() != 3 * iters) return;
  char what[160];
  for (int q = 0; q < 3 * iters; ++q) {
    std::snprintf(what, sizeof(what), "%s %dx%d units %d list %d", name, bm, bn, units, q);
    check_well_formed(pers[q], units, want[q % 3], what);
  }
  // causal: planning fewer iterations gives the same first lists
  const std::vector<TileList> two = plan_persistent(plan, bm, bn, kTcBK, units, 2);
  for (int q = 0; q < 6 && q < (int)two.size(); ++q)
    CHECK(same_lists(two[q], pers[q]), "%s: list %d depends on the planned iterations", name, q);
  // the waiting rules finish every tile, in any turn order and with any tile costs,
  // also for more iterations than were planned
  for (int seed = 0; seed < 3; ++seed) {
    const RunResult r = run_rules(plan, pers, units, 8, seed);
    CHECK(r.tiles_run == r.tiles_total, "%s: deadlock after %lld of %lld tiles (seed %d)", name,
          (long long)r.tiles_run, (long long)r.tiles_total, seed);
  }
  if (timed) {
    std::vector<TileList> matrix_order;
    for (int p = 0; p < 3; ++p)
      matrix_order.push_back(plan_tiles(plan, p, bm, bn, kTcBK, units, /*by_cost=*/false));
    for (TileList& tl : matrix_order)
      while ((int)tl.cta_begin.size() < units + 1) tl.cta_begin.push_back(tl.cta_begin.back());
    const RunResult a = run_rules(plan, pers, units, 5, -1);
    const RunResult b = run_rules(plan, matrix_order, units, 5, -1);
    CHECK(a.tiles_run == a.tiles_total && b.tiles_run == b.tiles_total, "%s: timed runs", name);
    CHECK(a.makespan <= b.makespan, "%s: simulated lists %.0f, matrix order %.0f", name,
          a.makespan, b.makespan);
    std::printf("%s %dx%d units %d: simulated lists %.0f, matrix order %.0f cost units\n", name,
                bm, bn, units, a.makespan, b.makespan);
  }
}

}  // namespace

int main() {
  Shapes gpt2, moe, ragged, one;
  for (int l = 0; l < 12; ++l)
    for (auto s : Shapes{{768, 2304}, {768, 768}, {768, 3072}, {3072, 768}}) gpt2.push_back(s);
  for (int e = 0; e < 16; ++e)
    for (auto s : Shapes{{2048, 1408}, {2048, 1408}, {1408, 2048}}) moe.push_back(s);
  ragged = {{300, 200}, {130, 520}, {200, 200}, {1, 50}, {7, 3}, {64, 1000}, {257, 129},
            {1, 1}, {384, 256}};
  one = {{256, 128}};
  check_set("gpt2", gpt2, 256, 256, 76, true);
  check_set("gpt2", gpt2, 128, 256, 152, true);
  check_set("moe16", moe, 256, 512, 76, false);
  check_set("ragged", ragged, 256, 256, 76, false);
  check_set("ragged", ragged, 128, 256, 5, false);
  check_set("one", one, 256, 256, 76, false);
  check_set("one", one, 128, 256, 1, false);
  if (g_failures == 0) std::printf("OK\n");
  return g_failures == 0 ? 0 : 1;
}
