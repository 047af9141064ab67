// Expert placement and replication planner (host code) for the expert-parallel layer.
//
// "Wide-EP ... MoE ... NVIDIA" explainer, section "Load imbalance: EPLB": between forward
// passes the per-expert load is inspected and the experts are re-placed; the most loaded
// experts get copies on several GPUs.  The page gives no algorithm; this is the plain
// greedy reading of it, fed by the per-expert token counts the permute produces:
//   1. replication: every expert starts with one copy; while free slots remain, one more
//      copy goes to the expert with the largest load per copy (ties: lower id), never
//      more copies than GPUs;
//   2. placement: copies, each carrying load / copies, are taken in descending load
//      (ties: lower expert id, then lower copy index) and put on the least loaded GPU that
//      still has a free slot and holds no copy of that expert (ties: lower GPU id); an
//      extra copy for which no such GPU is left is dropped (its share goes to the placed
//      copies: the loads are recomputed from the final copy counts).  An expert's first
//      copy always finds a slot, so every expert keeps at least one.
#include <algorithm>
#include <cstdint>
#include <vector>

#include "moe.h"

extern "C" moe_status moe_eplb_plan(const int64_t* load, int E, int G, int S, int32_t* slot_expert,
                                    int32_t* replicas, double* gpu_load) {
  if (!load || !slot_expert || !replicas || !gpu_load) return MOE_ERR_INVALID_ARG;
  if (E < 1 || G < 1 || S < 1 || static_cast<int64_t>(G) * S < E || static_cast<int64_t>(G) * S > (1 << 24))
    return MOE_ERR_INVALID_ARG;
  for (int e = 0; e < E; ++e)
    if (load[e] < 0) return MOE_ERR_INVALID_ARG;

  // 1. replication
  std::vector<int32_t> r(E, 1);
  int64_t used = E;
  const int64_t slots = static_cast<int64_t>(G) * S;
  while (used < slots) {
    int best = -1;
    for (int e = 0; e < E; ++e) {
      if (r[e] >= G) continue;
      // load[e] / r[e] > load[best] / r[best], compared exactly in integers
      if (best < 0 || static_cast<__int128>(load[e]) * r[best] > static_cast<__int128>(load[best]) * r[e]) best = e;
    }
    if (best < 0) break;  // every expert already has a copy on every GPU
    ++r[best];
    ++used;
  }

  // 2. placement, copies in descending per-copy load
  struct Copy {
    int e, c;
  };
  std::vector<Copy> copies;
  copies.reserve(used);
  for (int e = 0; e < E; ++e)
    for (int c = 0; c < r[e]; ++c) copies.push_back({e, c});
  std::stable_sort(copies.begin(), copies.end(), [&](const Copy& a, const Copy& b) {
    const __int128 lhs = static_cast<__int128>(load[a.e]) * r[b.e], rhs = static_cast<__int128>(load[b.e]) * r[a.e];
    if (lhs != rhs) return lhs > rhs;
    return a.e != b.e ? a.e < b.e : a.c < b.c;
  });
  std::vector<double> gl(G, 0.0);
  std::vector<int> fill(G, 0), placed(E, 0);
  std::vector<char> holds(static_cast<size_t>(G) * E, 0);
  for (int64_t i = 0; i < slots; ++i) slot_expert[i] = -1;
  for (const Copy& cp : copies) {
    int g_best = -1;
    for (int g = 0; g < G; ++g) {
      if (fill[g] >= S || holds[static_cast<size_t>(g) * E + cp.e]) continue;
      if (g_best < 0 || gl[g] < gl[g_best]) g_best = g;
    }
    if (g_best < 0) continue;  // extra copy with no GPU left to take it: dropped
    slot_expert[static_cast<int64_t>(g_best) * S + fill[g_best]] = cp.e;
    ++fill[g_best];
    ++placed[cp.e];
    holds[static_cast<size_t>(g_best) * E + cp.e] = 1;
    gl[g_best] += static_cast<double>(load[cp.e]) / r[cp.e];
  }
  // final loads from the placed copy counts
  for (int g = 0; g < G; ++g) {
    double sum = 0.0;
    for (int s = 0; s < S; ++s) {
      const int e = slot_expert[static_cast<int64_t>(g) * S + s];
      if (e >= 0) sum += static_cast<double>(load[e]) / placed[e];
    }
    gpu_load[g] = sum;
  }
  for (int e = 0; e < E; ++e) replicas[e] = placed[e];
  return MOE_OK;
}
